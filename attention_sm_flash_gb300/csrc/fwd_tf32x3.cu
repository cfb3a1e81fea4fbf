// fp32 attention forward on the tensor cores: tcgen05.mma kind::tf32 with a three-term
// split, TMA-staged tiles, accumulators in TMEM.
//
// The fp32 attention of the video pipeline's VAE runs on an fp32 CUTLASS kernel
// ("LingBot full-pipeline analysis report", section on the per-group shapes and
// attribution of the kernel ledger: fmha_cutlassF_f32 in vae_frame). TF32 products alone
// keep 10 mantissa bits, far from an fp32 result. Each fp32 operand x is split into
// hi = x rounded to TF32 and lo = x - hi (exact in fp32, itself TF32 to 2^-11 of lo), and
// each product into three tensor-core products,
//     a b ~ a_hi b_hi + a_hi b_lo + a_lo b_hi        (the a_lo b_lo term, ~2^-22 |a b|,
//                                                     is left out)
// accumulated in fp32: S = Q K^T and P V both this way. The tensor core's fp32
// accumulation rounds each step (measured: about 3e-6 absolute error on O after the
// ~2300 accumulating MMAs of a 6240-key row when O accumulated in TMEM across tiles), so
// the accumulation chains are kept short: within a product the small lo terms go first
// and the hi x hi terms last, and each key tile's P V lands in a fresh TMEM partial that
// the threads add into O with round-to-nearest fp32 arithmetic, O = alpha O + (P V)_tile,
// alpha the tile's rescale of the running max. The online softmax, masks and epilogue
// are those of the bf16 kernel (running max, rescale when it grows by more than 2^8, keys
// past the valid length masked and their V rows zeroed).
//
// One CTA of 256 threads per SM loops over items of 128 query rows of one (batch, head);
// the key tiles hold 64 keys. Phases, each closed by a CTA barrier:
//   Q tile (TMA) -> Q_hi in place in shared memory, Q_lo into TMEM (the A operand of
//   the third S term);
//   per key tile: K, V (TMA, issued as soon as the previous tile has finished with their
//   staging tiles) -> K_hi in place, K_lo beside it, V transposed to V^T (keys contiguous,
//   the K-major B operand of the PV products; keys run fastest across the threads, so
//   the transpose is free of bank conflicts) as hi and lo; S by 3 x D / 8 MMAs; softmax
//   (warps 0-3, one thread per row): P_hi over S's columns, P_lo beside it; the partial
//   T = P V by 3 x 8 MMAs with P from TMEM; O = alpha O + T by all eight warps (two per
//   TMEM lane quarter, half the columns each);
//   epilogue: O / l to global memory (fp32), LSE.
// (Running the V transpose under the S product and splitting the next K tile under the
// softmax was measured slower: 103 against 106.6 TFLOP/s on the fp32 DiT-frame case.)
// Every operand is K-major. Every wait is bounded in time; a wait that runs out flags
// ATTN_DEVERR_TIMEOUT and the CTA stops after letting its MMAs finish.

#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <mutex>

#include "attn_internal.h"
#include "fastdiv.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

using namespace sm103;

constexpr int kBM = 128;       // query rows of an item (TMEM lanes)
constexpr int kBN = 64;        // keys of a K/V tile
constexpr int kThreads = 256;  // warps 0-3 softmax + all phases; warps 4-7 the other phases
constexpr float kRescaleThreshold = 8.0f;

struct Tf32Params {
  CUtensorMap tm_q, tm_k, tm_v;
  float* o;
  float* lse;
  const int32_t* kv_lens;
  unsigned int* err;
  int B, Hq, Hkv, Sq, Skv, causal;
  int n_qblocks, n_items;
  FastDiv fd_qb, fd_hq, fd_g;
  float scale_log2;
  uint64_t timeout_ns;
};

struct Tf32Ctl {
  uint64_t tma_bar, mma_bar, k_bar, v_bar;  // Q; MMAs; the K and V tiles
  uint32_t tmem_base;
  int abort;
  float alpha[kBM];  // per row: the tile's rescale of O
};

// tcgen05.mma kind::tf32, D (+)= A B^T: A from shared memory or TMEM, B from shared memory
__device__ __forceinline__ void mma_tf32_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_tf32_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// Instruction descriptor of kind::tf32: fp32 accumulator (bits 4-5 = 1), TF32 A and B
// (bits 7-9 = 2, bits 10-12 = 2), both K-major, N >> 3 (bits 17-22), M >> 4 (bits 24-28).
constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// x rounded to TF32 (10 explicit mantissa bits, to nearest, ties away) as an fp32 value
__device__ __forceinline__ float tf32_hi(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u);
}

// Byte offset of element (row, col) in a tile of 32-bit elements stored as 128-byte rows
// of 32 columns, 128-byte swizzle, chunks of 32 columns `chunk_bytes` apart (the layout a
// TMA box of 32 columns x rows writes, and the K-major operand layout of tcgen05).
__device__ __forceinline__ uint32_t sw_off(int row, int col, int chunk_bytes) {
  return (uint32_t)((col >> 5) * chunk_bytes + row * 128 + ((((col & 31) >> 2) ^ (row & 7)) << 4) +
                    ((col & 3) << 2));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) fwd_tf32x3_kernel(const __grid_constant__ Tf32Params p) {
  constexpr int kQChunk = kBM * 128;   // 32 columns of the Q tile
  constexpr int kKChunk = kBN * 128;   // 32 columns of a K or V tile
  constexpr int kVTChunk = D * 128;    // 32 keys of a V^T tile
  constexpr int kQBytes = kBM * D * 4, kKBytes = kBN * D * 4;
  constexpr uint32_t kIdescS = idesc_tf32(kBM, kBN);
  constexpr uint32_t kIdescO = idesc_tf32(kBM, D);
  // TMEM columns: S, then P_hi over it [0, 64), P_lo [64, 128), O [128, 128 + D), the
  // tile's partial T = P V [128 + D, 128 + 2 D), Q_lo [128 + 2 D, 128 + 3 D)
  constexpr uint32_t kColPh = 0, kColPl = 64, kColO = 128, kColT = 128 + D, kColQl = 128 + 2 * D;
  static_assert(kColQl + D <= 512, "TMEM columns");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                   // Q_hi (in place of Q)
  uint8_t* sK = sQ + kQBytes;           // K_hi (in place of K)
  uint8_t* sKl = sK + kKBytes;          // K_lo
  uint8_t* sV = sKl + kKBytes;          // V as loaded
  uint8_t* sVT = sV + kKBytes;          // V_hi^T
  uint8_t* sVTl = sVT + kKBytes;        // V_lo^T
  Tf32Ctl& c = *reinterpret_cast<Tf32Ctl*>(sVTl + kKBytes);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quad = warp % 4, half = warp / 4;
  const int r = quad * 32 + lane;  // this thread's TMEM lane / query row of the tile
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;

  if (threadIdx.x == 0) {
    mbar_init(&c.tma_bar, 1);
    mbar_init(&c.mma_bar, 1);
    mbar_init(&c.k_bar, 1);
    mbar_init(&c.v_bar, 1);
    c.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&c.tmem_base, 512);
    tmem_relinquish();
  }
  if (p.kv_lens != nullptr && blockIdx.x == 0) {
    for (int e = threadIdx.x; e < p.B * p.Hkv; e += kThreads) {
      const int raw = __ldg(p.kv_lens + e);
      if (raw < 0 || raw > p.Skv) atomicOr(p.err, ATTN_DEVERR_KVLEN);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  WaitCtl wc{&c.abort, p.err, p.timeout_ns};
  uint32_t tma_ph = 0, mma_ph = 0, k_ph = 0, v_ph = 0;
  bool ok = true;
  bool mma_pending = false;  // an MMA commit this CTA has not waited for
  bool k_pending = false, v_pending = false, q_pending = false;  // thread 0: loads not waited for

  // a CTA-wide bounded wait; every thread ends with the same verdict
  auto wait_all = [&](uint64_t* bar, uint32_t& ph) -> bool {
    const bool mine = wait_phase(bar, ph, wc);
    ph ^= 1;
    return __syncthreads_and(mine ? 1 : 0) != 0;
  };

  for (int idx = blockIdx.x; ok && idx < p.n_items; idx += gridDim.x) {
    const int bh = p.fd_qb.div(idx);
    const int qb = idx - bh * p.n_qblocks;
    const int b = p.fd_hq.div(bh), h = bh - b * p.Hq;
    const int kvh = p.fd_g.div(h);
    const int q0 = qb * kBM;
    int L = p.Skv;
    if (p.kv_lens != nullptr) {
      L = __ldg(p.kv_lens + b * p.Hkv + kvh);
      L = L < 0 ? 0 : (L > p.Skv ? p.Skv : L);
    }
    int kmax = L;
    if (p.causal) kmax = min(L, min(q0 + kBM - 1, p.Sq - 1) + L - p.Sq + 1);
    kmax = max(kmax, 0);
    const int n = (kmax + kBN - 1) / kBN;
    const int i = q0 + r;
    const bool row_ok = half == 0 && i < p.Sq;
    float* orow = p.o + ((static_cast<int64_t>(b) * p.Sq + i) * p.Hq + h) * D;
    float* lrow = p.lse + (static_cast<int64_t>(b) * p.Hq + h) * p.Sq + i;
    if (n == 0) {
      if (row_ok) {
        for (int d = 0; d < D; d += 4) *reinterpret_cast<float4*>(orow + d) = make_float4(0.f, 0.f, 0.f, 0.f);
        *lrow = -CUDART_INF_F;
      }
      continue;
    }
    // ---- Q: TMA, then Q_hi in place and Q_lo into TMEM (this thread's row, half the columns)
    // K(j) and V(j) into their staging tiles; tile j + 1's loads start as soon as tile j
    // has finished with them (V after its transpose, K after the S product)
    auto load_k = [&](int jj) {
      mbar_expect_tx(&c.k_bar, kKBytes);
      for (int ch = 0; ch < D / 32; ++ch) tma_load_4d(sK + ch * kKChunk, &p.tm_k, &c.k_bar, ch * 32, kvh, jj * kBN, b);
    };
    auto load_v = [&](int jj) {
      mbar_expect_tx(&c.v_bar, kKBytes);
      for (int ch = 0; ch < D / 32; ++ch) tma_load_4d(sV + ch * kKChunk, &p.tm_v, &c.v_bar, ch * 32, kvh, jj * kBN, b);
    };
    if (threadIdx.x == 0) {
      mbar_expect_tx(&c.tma_bar, kQBytes);
      for (int ch = 0; ch < D / 32; ++ch) tma_load_4d(sQ + ch * kQChunk, &p.tm_q, &c.tma_bar, ch * 32, h, q0, b);
      load_k(0);
      load_v(0);
      k_pending = v_pending = q_pending = true;
    }
    if (!wait_all(&c.tma_bar, tma_ph)) { ok = false; break; }
    q_pending = false;
#pragma unroll 1
    for (int c0 = half * (D / 2); c0 < half * (D / 2) + D / 2; c0 += 32) {
      uint32_t lo[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        float* a = reinterpret_cast<float*>(sQ + sw_off(r, c0 + e, kQChunk));
        const float x = *a, hi = tf32_hi(x);
        *a = hi;
        lo[e] = __float_as_uint(x - hi);
      }
      tmem_st32(tmem + lane_off + kColQl + c0, lo);
    }
    tmem_wait_st();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const int kend = p.causal ? min(L, i + L - p.Sq + 1) : L;  // keys visible to row i
    float m = -CUDART_INF_F, l = 0.f;
    float alpha = 1.f;  // this tile's rescale of O (softmax threads; shared below)
    for (int j = 0; ok && j < n; ++j) {
      // ---- K, V of tile j
      if (!wait_all(&c.k_bar, k_ph)) { ok = false; break; }
      k_pending = false;
      if (!wait_all(&c.v_bar, v_ph)) { ok = false; break; }
      v_pending = false;
      // K_hi in place, K_lo beside it (the layout is element-wise, any order works)
      for (int e = threadIdx.x; e < kKBytes / 16; e += kThreads) {
        float4* a = reinterpret_cast<float4*>(sK) + e;
        const float4 x = *a;
        const float4 hi = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
        *a = hi;
        reinterpret_cast<float4*>(sKl)[e] = make_float4(x.x - hi.x, x.y - hi.y, x.z - hi.z, x.w - hi.w);
      }
      // V^T (keys contiguous), hi and lo; keys at or past the valid length are zero, so
      // padding (even NaN) never meets P = 0 in a product
      for (int e = threadIdx.x; e < kBN * D / 4; e += kThreads) {
        const int key = e % kBN, d0 = (e / kBN) * 4;
        float4 x = *reinterpret_cast<const float4*>(sV + sw_off(key, d0, kKChunk));
        if (j * kBN + key >= L) x = make_float4(0.f, 0.f, 0.f, 0.f);
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float hi = tf32_hi(xs[t]);
          const uint32_t o = sw_off(d0 + t, key, kVTChunk);
          *reinterpret_cast<float*>(sVT + o) = hi;
          *reinterpret_cast<float*>(sVTl + o) = xs[t] - hi;
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0 && j + 1 < n) {
        load_v(j + 1);
        v_pending = true;
      }
      // ---- S = Q K^T, three terms per 8-wide step of D
      if (threadIdx.x == 0) {
        tc_fence_after();
        const uint64_t dq = smem_desc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dk = smem_desc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t dkl = smem_desc_sw128(smem_u32(sKl), 16, 1024);
        // the small terms first (the accumulator stays small while they are added), then
        // hi x hi
#pragma unroll
        for (int kk = 0; kk < D / 8; ++kk) {
          const uint32_t oq = ((kk / 4) * kQChunk + (kk % 4) * 32) >> 4;
          const uint32_t ok_ = ((kk / 4) * kKChunk + (kk % 4) * 32) >> 4;
          mma_tf32_ss(tmem, dq + oq, dkl + ok_, kIdescS, kk > 0 ? 1u : 0u);
          mma_tf32_ts(tmem, tmem + kColQl + kk * 8, dk + ok_, kIdescS, 1u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 8; ++kk) {
          const uint32_t oq = ((kk / 4) * kQChunk + (kk % 4) * 32) >> 4;
          const uint32_t ok_ = ((kk / 4) * kKChunk + (kk % 4) * 32) >> 4;
          mma_tf32_ss(tmem, dq + oq, dk + ok_, kIdescS, 1u);
        }
        mma_commit(&c.mma_bar);
      }
      if (!wait_all(&c.mma_bar, mma_ph)) { ok = false; break; }
      tc_fence_after();
      if (threadIdx.x == 0 && j + 1 < n) {
        load_k(j + 1);
        k_pending = true;
      }
      // ---- softmax (warps 0-3, one row each); warps 4-7 wait at the barrier below
      if (half == 0) {
        float s[kBN];
        tmem_ld64(tmem + lane_off, reinterpret_cast<uint32_t*>(s));
        const int limit = kend - j * kBN;
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int e = 0; e < kBN; ++e) {
          s[e] = e < limit ? s[e] * p.scale_log2 : -CUDART_INF_F;
          mx = fmaxf(mx, s[e]);
        }
        const float mnew = fmaxf(m, mx);
        alpha = 1.f;
        if (mnew > m + kRescaleThreshold) {
          // O (the sum through the previous tile) is scaled by alpha when T is added
          if (m != -CUDART_INF_F) {
            alpha = ex2_approx(m - mnew);
            l *= alpha;
          }
          m = mnew;
        }
        const float msub = m == -CUDART_INF_F ? 0.f : m;
#pragma unroll
        for (int q2 = 0; q2 < kBN / 32; ++q2) {
          uint32_t ph[32], pl[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float pe = ex2_approx(s[q2 * 32 + e] - msub);  // 0 where masked
            l += pe;
            const float hi = tf32_hi(pe);
            ph[e] = __float_as_uint(hi);
            pl[e] = __float_as_uint(pe - hi);
          }
          tmem_st32(tmem + lane_off + kColPh + q2 * 32, ph);
          tmem_st32(tmem + lane_off + kColPl + q2 * 32, pl);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncthreads();
      // ---- O += P V, three terms per 8-key step
      if (threadIdx.x == 0) {
        tc_fence_after();
        const uint64_t dv = smem_desc_sw128(smem_u32(sVT), 16, 1024);
        const uint64_t dvl = smem_desc_sw128(smem_u32(sVTl), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 8; ++kk) {
          const uint32_t ov = ((kk / 4) * kVTChunk + (kk % 4) * 32) >> 4;
          mma_tf32_ts(tmem + kColT, tmem + kColPh + kk * 8, dvl + ov, kIdescO, kk > 0 ? 1u : 0u);
          mma_tf32_ts(tmem + kColT, tmem + kColPl + kk * 8, dv + ov, kIdescO, 1u);
        }
#pragma unroll
        for (int kk = 0; kk < kBN / 8; ++kk) {
          const uint32_t ov = ((kk / 4) * kVTChunk + (kk % 4) * 32) >> 4;
          mma_tf32_ts(tmem + kColT, tmem + kColPh + kk * 8, dv + ov, kIdescO, 1u);
        }
        mma_commit(&c.mma_bar);
      }
      mma_pending = true;
      if (!wait_all(&c.mma_bar, mma_ph)) { ok = false; break; }
      mma_pending = false;
      tc_fence_after();
      // ---- O = alpha O + T: both warps of a lane quarter, half the columns each; the
      // softmax warp of the quarter hands its rows' alpha to the other through shared memory
      if (half == 0) c.alpha[r] = alpha;
      __syncthreads();
      {
        const float a = c.alpha[r];
#pragma unroll 1
        for (int cc = half * (D / 64); cc < (half + 1) * (D / 64); ++cc) {
          uint32_t tv[32];
          tmem_ld32(tmem + lane_off + kColT + cc * 32, tv);
          if (j == 0) {
            tmem_st32(tmem + lane_off + kColO + cc * 32, tv);
          } else {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_off + kColO + cc * 32, ov);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              ov[e] = __float_as_uint(__fmaf_rn(__uint_as_float(ov[e]), a, __uint_as_float(tv[e])));
            tmem_st32(tmem + lane_off + kColO + cc * 32, ov);
          }
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
    if (!ok) break;
    // ---- epilogue: O / l, LSE
    if (half == 0) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t ov[32];
        tmem_ld32(tmem + lane_off + kColO + cc * 32, ov);
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(orow + cc * 32 + e) =
                make_float4(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv,
                            __uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv);
        }
      }
      if (row_ok) *lrow = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  // an MMA whose completion was not waited for (a wait that ran out) must finish before
  // the TMEM is freed
  if (threadIdx.x == 0 && (mma_pending || !ok)) {
    mma_commit(&c.mma_bar);
    wait_phase_teardown(&c.mma_bar, mma_ph, 200000000ull);
  }
  if (threadIdx.x == 0 && k_pending) wait_phase_teardown(&c.k_bar, k_ph, 200000000ull);
  if (threadIdx.x == 0 && v_pending) wait_phase_teardown(&c.v_bar, v_ph, 200000000ull);
  if (threadIdx.x == 0 && q_pending) wait_phase_teardown(&c.tma_bar, tma_ph, 200000000ull);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// An fp32 [B, S, H, D] tensor as a 4-D TMA map (D, H, S, B) whose box is one head: 32
// columns (128 bytes, 128-byte swizzle) x `rows` tokens.
bool make_f32_map(CUtensorMap* map, const void* base, int B, int S, int H, int D, int rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4, (cuuint64_t)S * H * D * 4};
  const cuuint32_t box[4] = {32, 1, (cuuint32_t)rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
constexpr size_t tf32_smem_bytes() {
  return 1024 + (size_t)kBM * D * 4 + 5 * (size_t)kBN * D * 4 + sizeof(Tf32Ctl);
}

constexpr int kMaxDev = 64;
std::mutex g_mu;
int g_num_sms[kMaxDev] = {};
bool g_attr_set[kMaxDev][2] = {};

template <int D>
cudaError_t launch_tf32(const Tf32Params& prm, int dev, cudaStream_t s) {
  constexpr size_t smem = tf32_smem_bytes<D>();
  static_assert(smem <= 232448, "shared memory per block");
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_attr_set[dev][D == 64 ? 0 : 1]) {
      cudaError_t e = cudaFuncSetAttribute(fwd_tf32x3_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      g_attr_set[dev][D == 64 ? 0 : 1] = true;
    }
  }
  const int grid = prm.n_items < g_num_sms[dev] ? prm.n_items : g_num_sms[dev];
  fwd_tf32x3_kernel<D><<<grid, kThreads, smem, s>>>(prm);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tf32_fwd(const Problem& p, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_num_sms[dev] == 0) {
      e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
    }
  }
  Tf32Params prm{};
  const bool no_keys = p.Skv == 0;
  if (!make_f32_map(&prm.tm_q, p.q, p.B, p.Sq, p.Hq, p.D, kBM) ||
      !make_f32_map(&prm.tm_k, no_keys ? p.q : p.k, p.B, no_keys ? p.Sq : p.Skv, no_keys ? p.Hq : p.Hkv, p.D, kBN) ||
      !make_f32_map(&prm.tm_v, no_keys ? p.q : p.v, p.B, no_keys ? p.Sq : p.Skv, no_keys ? p.Hq : p.Hkv, p.D, kBN))
    return cudaErrorInvalidValue;
  prm.o = static_cast<float*>(p.o);
  prm.lse = p.lse;
  prm.kv_lens = p.kv_lens;
  prm.err = p.err;
  prm.B = p.B;
  prm.Hq = p.Hq;
  prm.Hkv = p.Hkv;
  prm.Sq = p.Sq;
  prm.Skv = p.Skv;
  prm.causal = p.causal;
  prm.n_qblocks = (p.Sq + kBM - 1) / kBM;
  prm.n_items = p.B * p.Hq * prm.n_qblocks;
  prm.fd_qb = FastDiv::make(prm.n_qblocks);
  prm.fd_hq = FastDiv::make(p.Hq);
  prm.fd_g = FastDiv::make(p.Hq / p.Hkv);
  prm.scale_log2 = p.scale * 1.4426950408889634f;
  prm.timeout_ns = 4000000000ull;
  return p.D == 64 ? launch_tf32<64>(prm, dev, s) : launch_tf32<128>(prm, dev, s);
}

}  // namespace attn
