// bf16 attention backward for sm_103a: tcgen05 MMAs into TMEM, TMA-staged tiles.
//
// The flash backward of "xtrain evolution.md" (infrastructure table, row T14): the
// scores are recomputed from Q, K and the forward's LSE, delta = rowsum(dO * O) (computed
// beforehand into the caller's workspace) simplifies the softmax Jacobian:
//     P = exp(scale * Q K^T - LSE),  dP = dO V^T,  dS = P * (dP - delta),
//     dV = P^T dO,  dK = scale * dS^T Q,  dQ = scale * dS K.
// Two kernels, both deterministic (every sum in a fixed order, no atomics):
//
// dK/dV: a CTA owns 128 keys of one (batch, kv head) and loops over the query heads of
//   the GQA group and their query tiles of 64 rows in a fixed order, so the group sum of
//   row T15 (in-group deterministic sum) happens inside its TMEM accumulators. When such
//   items are too few to fill the GPU (few kv heads, causal imbalance), each query head
//   is its own item writing fp32 partial dK/dV, and a reduction kernel sums each group
//   in head order - still deterministic, still no atomics. Keys sit
//   on the TMEM lanes: S^T = K Q^T and dP^T = V dO^T (M = 128 keys, N = 64 queries), the
//   elementwise warps turn them into P^T and dS^T (bf16, written back over the first
//   half of the same columns), then dV += P^T dO and dK += dS^T Q with A from TMEM.
//   S^T/dP^T are double-buffered, so the elementwise work of one query tile overlaps
//   the MMAs of the next.
// dQ: a CTA owns 128 query rows of one (batch, head) and loops over K/V tiles of 64
//   keys: S = Q K^T, dP = dO V^T, dS on the elementwise warps, dQ += dS K.
//
// Roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer (one thread), warps 2-5
// and 6-9 two elementwise warpgroups taking alternate tiles (warp w reaches the TMEM
// lanes 32 * (w % 4) ..). Every barrier wait is
// bounded in time; a wait that runs out flags ATTN_DEVERR_TIMEOUT and the CTA gives up
// after letting its copies and MMAs in flight finish.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <mutex>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

using namespace sm103;

constexpr int kThreads = 320;  // warps 0-1: producer, MMA; warps 2-5, 6-9: elementwise
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kTeardownNs = 200000000ull;

struct BwdParams {
  CUtensorMap tm_q, tm_do, tm_k, tm_v;
  const float* lse;
  const float* delta;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* part_dk;  // split mode: fp32 per-query-head partial dK, dV [B, Skv, Hq, D]
  float* part_dv;
  const int32_t* kv_lens;
  unsigned int* err;
  int B, Hq, Hkv, Sq, Skv, causal;
  int split;
  int n_items;
  float scale, scale_log2;
  uint64_t timeout_ns;
};

__device__ __forceinline__ int kv_len_of(const BwdParams& p, int b, int kvh) {
  if (p.kv_lens == nullptr) return p.Skv;
  const int L = __ldg(p.kv_lens + b * p.Hkv + kvh);
  return L < 0 ? 0 : (L > p.Skv ? p.Skv : L);
}

__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const uint32_t* v, float mul) {
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e)
    pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int e = 0; e < 4; ++e) d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
}

__device__ __forceinline__ void zero_row_bf16(__nv_bfloat16* dst, int n) {
  for (int d = 0; d < n; d += 8) *reinterpret_cast<uint4*>(dst + d) = make_uint4(0u, 0u, 0u, 0u);
}

// =============================================================================== dK/dV
constexpr int kKeys = 128;  // keys per CTA item (TMEM lanes)
constexpr int kQT = 64;     // queries per tile

template <int NST>
struct DkvCtl {
  uint64_t kv_full, kv_empty, acc_done, acc_free, mma_final;
  uint64_t st_full[NST], st_empty[NST];
  uint64_t sp_full[2], ds_ready[2], mm2_done[2];
  uint32_t tmem_base;
  int abort;
  float lse[NST][kQT];  // LSE * log2(e) of the tile's queries (+inf: no contribution)
  float del[NST][kQT];
};

struct DkvItem {
  int b, kvh, j0, L;
  int h0, heads;  // query heads h0 .. h0 + heads - 1 (the whole group, or one in split mode)
  int i_start, per_head, n_tiles;
};

__device__ __forceinline__ DkvItem dkv_decode(int idx, const BwdParams& p) {
  const int n_kt = (p.Skv + kKeys - 1) / kKeys;
  const int g = p.Hq / p.Hkv;
  const int gs = p.split ? g : 1;  // items per (batch, kv head, key tile)
  const int BK = p.B * p.Hkv;
  int b, kvh, kt, r;
  if (p.causal) {
    // longest first: the first key tiles are seen by the most queries
    kt = idx / (BK * gs);
    const int rem = idx % (BK * gs);
    const int bk = rem / gs;
    r = rem % gs;
    b = bk / p.Hkv;
    kvh = bk % p.Hkv;
  } else {
    const int bk = idx / (n_kt * gs);
    const int rem = idx % (n_kt * gs);
    kt = rem / gs;
    r = rem % gs;
    b = bk / p.Hkv;
    kvh = bk % p.Hkv;
  }
  DkvItem it;
  it.b = b;
  it.kvh = kvh;
  it.j0 = kt * kKeys;
  it.L = kv_len_of(p, b, kvh);
  it.h0 = kvh * g + r;
  it.heads = p.split ? 1 : g;
  const int n_qt = (p.Sq + kQT - 1) / kQT;
  it.i_start = 0;
  it.per_head = 0;
  if (it.j0 < it.L) {
    // queries that see key j0: i >= j0 - L + Sq (causal, bottom-right)
    const int first = p.causal ? max(0, it.j0 - it.L + p.Sq) : 0;
    it.i_start = first / kQT;
    it.per_head = max(0, n_qt - it.i_start);
  }
  it.n_tiles = it.heads * it.per_head;
  return it;
}

template <int D, int NST>
__global__ void __launch_bounds__(kThreads, 1) bwd_dkdv_sm103_kernel(const __grid_constant__ BwdParams p) {
  constexpr int kKTile = kKeys * D * 2;  // K or V tile bytes
  constexpr int kKChunk = kKeys * 128;
  constexpr int kQTile = kQT * D * 2;    // Q or dO tile bytes
  constexpr int kQChunk = kQT * 128;
  constexpr int kChunks = D / 64;
  constexpr uint32_t kIdescSP = idesc_bf16_f32(kKeys, kQT, false, false);
  constexpr uint32_t kIdescAcc = idesc_bf16_f32(kKeys, D, false, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + kKTile;
  uint8_t* sQ = smem + 2 * kKTile;                 // NST stages
  uint8_t* sdO = smem + 2 * kKTile + NST * kQTile;  // NST stages
  DkvCtl<NST>& c = *reinterpret_cast<DkvCtl<NST>*>(smem + 2 * kKTile + 2 * NST * kQTile);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = p.Hq / p.Hkv;

  if (threadIdx.x == 0) {
    mbar_init(&c.kv_full, 1);
    mbar_init(&c.kv_empty, 1);
    mbar_init(&c.acc_done, 1);
    mbar_init(&c.acc_free, 256);
    mbar_init(&c.mma_final, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&c.st_full[s], 2);  // TMA (expect_tx) + LSE/delta stores
      mbar_init(&c.st_empty[s], 1);
    }
    for (int u = 0; u < 2; ++u) {
      mbar_init(&c.sp_full[u], 1);
      mbar_init(&c.ds_ready[u], 128);
      mbar_init(&c.mm2_done[u], 1);
    }
    c.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
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
  const uint32_t t_dv = tmem, t_dk = tmem + D;
  WaitCtl wc{&c.abort, p.err, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    uint32_t kv_cnt = 0, st = 0, st_par = 0, issued = 0, last_par = 0;
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < p.n_items; idx += gridDim.x) {
      const DkvItem it = dkv_decode(idx, p);
      if (it.n_tiles == 0) continue;
      if (!wait_phase_warp(&c.kv_empty, (kv_cnt & 1) ^ 1, wc)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(&c.kv_full, 2 * kKTile);
        for (int ch = 0; ch < kChunks; ++ch) {
          tma_load_4d(sK + ch * kKChunk, &p.tm_k, &c.kv_full, ch * 64, it.kvh, it.j0, it.b);
          tma_load_4d(sV + ch * kKChunk, &p.tm_v, &c.kv_full, ch * 64, it.kvh, it.j0, it.b);
        }
      }
      ++kv_cnt;
      for (int t = 0; t < it.n_tiles; ++t) {
        const int h = it.h0 + t / it.per_head;
        const int i0 = (it.i_start + t % it.per_head) * kQT;
        if (!wait_phase_warp(&c.st_empty[st], st_par ^ 1, wc)) { ok = false; break; }
        if (lane == 0) {
          mbar_expect_tx(&c.st_full[st], 2 * kQTile);
          for (int ch = 0; ch < kChunks; ++ch) {
            tma_load_4d(sQ + st * kQTile + ch * kQChunk, &p.tm_q, &c.st_full[st], ch * 64, h, i0, it.b);
            tma_load_4d(sdO + st * kQTile + ch * kQChunk, &p.tm_do, &c.st_full[st], ch * 64, h, i0, it.b);
          }
        }
        issued |= 1u << st;
        last_par = (last_par & ~(1u << st)) | (st_par << st);
        const int64_t row0 = (static_cast<int64_t>(it.b) * p.Hq + h) * p.Sq;
#pragma unroll
        for (int k2 = 0; k2 < kQT / 32; ++k2) {
          const int q = lane + 32 * k2;
          const int i = i0 + q;
          float l2 = CUDART_INF_F, dl = 0.f;
          if (i < p.Sq) {
            const float lv = __ldg(p.lse + row0 + i);
            // a row with no visible key (LSE = -inf) contributes nothing
            l2 = lv == -CUDART_INF_F ? CUDART_INF_F : lv * kLog2e;
            dl = __ldg(p.delta + row0 + i);
          }
          c.lse[st][q] = l2;
          c.del[st][q] = dl;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.st_full[st]);
        if (++st == NST) { st = 0; st_par ^= 1; }
      }
    }
    for (int s = 0; s < NST; ++s)
      if (issued & (1u << s)) wait_phase_teardown(&c.st_full[s], (last_par >> s) & 1, kTeardownNs);
    if (kv_cnt > 0) wait_phase_teardown(&c.kv_full, (kv_cnt - 1) & 1, kTeardownNs);
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t sKa = smem_u32(sK), sVa = smem_u32(sV);
      const uint32_t sQa = smem_u32(sQ), sdOa = smem_u32(sdO);
      uint32_t kv_cnt = 0, st = 0, st_par = 0, gt = 0, item_cnt = 0;
      bool ok = true;
      // dV += P^T dO and dK += dS^T Q for tile `tg` held in stage `s`
      auto acc_mmas = [&](uint32_t tg, uint32_t s, bool first) -> bool {
        const uint32_t u = tg & 1, cu = tg >> 1;
        if (!wait_phase(&c.ds_ready[u], cu & 1, wc)) return false;
        if (first && !wait_phase(&c.acc_free, (item_cnt & 1) ^ 1, wc)) return false;
        tc_fence_after();
        const uint32_t tbuf = tmem + 2 * D + u * 128;
#pragma unroll
        for (int kk = 0; kk < kQT / 16; ++kk) {
          const uint32_t acc = (first && kk == 0) ? 0u : 1u;
          const uint64_t bdo = smem_desc_sw128(sdOa + s * kQTile + kk * 16 * 128, kQChunk, 1024);
          mma_ts(t_dv, tbuf + kk * 8, bdo, kIdescAcc, acc);
          const uint64_t bq = smem_desc_sw128(sQa + s * kQTile + kk * 16 * 128, kQChunk, 1024);
          mma_ts(t_dk, tbuf + 64 + kk * 8, bq, kIdescAcc, acc);
        }
        mma_commit(&c.mm2_done[u]);
        mma_commit(&c.st_empty[s]);
        return true;
      };
      for (int idx = blockIdx.x; ok && idx < p.n_items; idx += gridDim.x) {
        const DkvItem it = dkv_decode(idx, p);
        if (it.n_tiles == 0) continue;
        if (!wait_phase(&c.kv_full, kv_cnt & 1, wc)) { ok = false; break; }
        tc_fence_after();
        uint32_t prev_st = 0;
        for (int t = 0; t < it.n_tiles; ++t) {
          const uint32_t u = gt & 1, cu = gt >> 1;
          if (!wait_phase(&c.st_full[st], st_par, wc)) { ok = false; break; }
          // buffer u holds P^T/dS^T of tile gt-2 until its accumulation MMAs complete
          if (cu >= 1 && !wait_phase(&c.mm2_done[u], (cu - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tbuf = tmem + 2 * D + u * 128;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * 0 + (kk % 4) * 32;
            const uint64_t ak = smem_desc_sw128(sKa + (kk / 4) * kKChunk + off, 16, 1024);
            const uint64_t bq = smem_desc_sw128(sQa + st * kQTile + (kk / 4) * kQChunk + off, 16, 1024);
            mma_ss(tbuf, ak, bq, kIdescSP, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk % 4) * 32;
            const uint64_t av = smem_desc_sw128(sVa + (kk / 4) * kKChunk + off, 16, 1024);
            const uint64_t bdo = smem_desc_sw128(sdOa + st * kQTile + (kk / 4) * kQChunk + off, 16, 1024);
            mma_ss(tbuf + 64, av, bdo, kIdescSP, kk > 0 ? 1u : 0u);
          }
          mma_commit(&c.sp_full[u]);
          if (t >= 1 && !acc_mmas(gt - 1, prev_st, t == 1)) { ok = false; break; }
          prev_st = st;
          if (++st == NST) { st = 0; st_par ^= 1; }
          ++gt;
        }
        if (!ok) break;
        if (!acc_mmas(gt - 1, prev_st, it.n_tiles == 1)) { ok = false; break; }
        mma_commit(&c.acc_done);
        mma_commit(&c.kv_empty);
        ++kv_cnt;
        ++item_cnt;
      }
      mma_commit(&c.mma_final);
      wait_phase_teardown(&c.mma_final, 0, kTeardownNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- elementwise
    const int w = (warp - 2) / 4;
    const int quad = warp % 4;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t gt = 0, item_cnt = 0;
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < p.n_items; idx += gridDim.x) {
      const DkvItem it = dkv_decode(idx, p);
      const int j = it.j0 + r;
      const bool key_ok = j < it.L;
      const int64_t orow = ((static_cast<int64_t>(it.b) * p.Skv + j) * p.Hkv + it.kvh) * D;
      if (it.n_tiles == 0) {
        if (j < p.Skv) {
          if (p.split) {
            float4* z = reinterpret_cast<float4*>((w == 0 ? p.part_dv : p.part_dk) +
                                                  ((static_cast<int64_t>(it.b) * p.Skv + j) * p.Hq + it.h0) * D);
            for (int d = 0; d < D / 4; ++d) z[d] = make_float4(0.f, 0.f, 0.f, 0.f);
          } else {
            zero_row_bf16((w == 0 ? p.dv : p.dk) + orow, D);
          }
        }
        continue;
      }
      for (int t = 0; t < it.n_tiles; ++t, ++gt) {
        if (static_cast<int>(gt & 1) != w) continue;
        const uint32_t s = gt % NST;
        if (!wait_phase_warp(&c.st_full[s], (gt / NST) & 1, wc)) { ok = false; break; }
        if (!wait_phase_warp(&c.sp_full[w], (gt >> 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tbuf = tmem + lane_off + 2 * D + w * 128;
        const int i0 = (it.i_start + t % it.per_head) * kQT;
        // causal: key j is visible to query i0 + q iff q >= j - L + Sq - i0
        const int qlo = p.causal ? j - it.L + p.Sq - i0 : -1;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pp[16], dd[16];
          float sv[32], dp[32];
          tmem_ld32(tbuf + half * 32, reinterpret_cast<uint32_t*>(sv));
          tmem_ld32(tbuf + 64 + half * 32, reinterpret_cast<uint32_t*>(dp));
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float pv[2], dv2[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int q = half * 32 + 2 * e + h2;
              const bool vis = key_ok && q >= qlo;
              const float x = fmaf(sv[2 * e + h2], p.scale_log2, -c.lse[s][q]);
              const float pq = vis ? ex2_approx(x) : 0.f;
              pv[h2] = pq;
              dv2[h2] = vis ? pq * (dp[2 * e + h2] - c.del[s][q]) : 0.f;
            }
            pp[e] = pack_bf16x2(pv[0], pv[1]);
            dd[e] = pack_bf16x2(dv2[0], dv2[1]);
          }
          // P^T over S^T's columns [16 half, ..), dS^T over dP^T's
          tmem_st16(tbuf + half * 16, pp);
          tmem_st16(tbuf + 64 + half * 16, dd);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&c.ds_ready[w]);
      }
      if (!ok) break;
      // epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK (times the scale)
      if (!wait_phase_warp(&c.acc_done, item_cnt & 1, wc)) { ok = false; break; }
      tc_fence_after();
      __nv_bfloat16* dst = (w == 0 ? p.dv : p.dk) + orow;
      float* pdst = (w == 0 ? p.part_dv : p.part_dk) +
                    ((static_cast<int64_t>(it.b) * p.Skv + j) * p.Hq + it.h0) * D;
      const uint32_t tacc = tmem + lane_off + (w == 0 ? 0 : D);
      const float mul = w == 0 ? 1.f : p.scale;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        tmem_ld32(tacc + cc * 32, v);
        if (j < p.Skv) {
          if (p.split) {
            // this query head's share, unscaled; the group reduction scales dK
            float4* d4 = reinterpret_cast<float4*>(pdst + cc * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              d4[e] = key_ok ? make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                           __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
          } else if (key_ok) {
            store_row_bf16(dst + cc * 32, v, mul);
          } else {
            zero_row_bf16(dst + cc * 32, 32);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&c.acc_free);
      ++item_cnt;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================================== dQ
constexpr int kQRows = 128;  // query rows per CTA item (TMEM lanes)
constexpr int kKT = 64;      // keys per tile

template <int NST>
struct DqCtl {
  uint64_t q_full, q_empty, acc_done, acc_free, mma_final;
  uint64_t st_full[NST], st_empty[NST], st_fixed[NST];
  uint64_t sp_full[2], ds_ready[2], mm2_done[2];
  uint32_t tmem_base;
  int abort;
};

struct DqItem {
  int b, h, kvh, q0, L, n_tiles;
};

__device__ __forceinline__ DqItem dq_decode(int idx, const BwdParams& p) {
  const int n_qt = (p.Sq + kQRows - 1) / kQRows;
  const int BH = p.B * p.Hq;
  int b, h, qt;
  if (p.causal) {
    qt = n_qt - 1 - idx / BH;  // longest first
    const int bh = idx % BH;
    b = bh / p.Hq;
    h = bh % p.Hq;
  } else {
    const int bh = idx / n_qt;
    qt = idx % n_qt;
    b = bh / p.Hq;
    h = bh % p.Hq;
  }
  DqItem it;
  it.b = b;
  it.h = h;
  it.kvh = h / (p.Hq / p.Hkv);
  it.q0 = qt * kQRows;
  it.L = kv_len_of(p, b, it.kvh);
  int kmax = it.L;
  if (p.causal) {
    const int ilast = min(it.q0 + kQRows - 1, p.Sq - 1);
    kmax = min(it.L, ilast + it.L - p.Sq + 1);
  }
  kmax = max(kmax, 0);
  it.n_tiles = (kmax + kKT - 1) / kKT;
  return it;
}

// K tile j holds in-bounds rows at or past the valid length (padding, maybe NaN); they
// are zeroed before dQ += dS K reads them.
__device__ __forceinline__ bool dq_needs_fix(int j, int L, int Skv) {
  return min(Skv, (j + 1) * kKT) > L;
}

template <int D, int NST>
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_sm103_kernel(const __grid_constant__ BwdParams p) {
  constexpr int kQTile = kQRows * D * 2;
  constexpr int kQChunk = kQRows * 128;
  constexpr int kKTile = kKT * D * 2;
  constexpr int kKChunk = kKT * 128;
  constexpr int kChunks = D / 64;
  constexpr uint32_t kIdescSP = idesc_bf16_f32(kQRows, kKT, false, false);
  constexpr uint32_t kIdescAcc = idesc_bf16_f32(kQRows, D, false, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sdO = smem + kQTile;
  uint8_t* sK = smem + 2 * kQTile;                  // NST stages
  uint8_t* sV = smem + 2 * kQTile + NST * kKTile;   // NST stages
  DqCtl<NST>& c = *reinterpret_cast<DqCtl<NST>*>(smem + 2 * kQTile + 2 * NST * kKTile);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(&c.q_full, 1);
    mbar_init(&c.q_empty, 1);
    mbar_init(&c.acc_done, 1);
    mbar_init(&c.acc_free, 256);
    mbar_init(&c.mma_final, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&c.st_full[s], 1);
      mbar_init(&c.st_empty[s], 1);
      mbar_init(&c.st_fixed[s], 1);
    }
    for (int u = 0; u < 2; ++u) {
      mbar_init(&c.sp_full[u], 1);
      mbar_init(&c.ds_ready[u], 128);
      mbar_init(&c.mm2_done[u], 1);
    }
    c.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&c.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  WaitCtl wc{&c.abort, p.err, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    uint32_t q_cnt = 0, st = 0, st_par = 0, issued = 0, last_par = 0;
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < p.n_items; idx += gridDim.x) {
      const DqItem it = dq_decode(idx, p);
      if (it.n_tiles == 0) continue;
      if (!wait_phase_warp(&c.q_empty, (q_cnt & 1) ^ 1, wc)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(&c.q_full, 2 * kQTile);
        for (int ch = 0; ch < kChunks; ++ch) {
          tma_load_4d(sQ + ch * kQChunk, &p.tm_q, &c.q_full, ch * 64, it.h, it.q0, it.b);
          tma_load_4d(sdO + ch * kQChunk, &p.tm_do, &c.q_full, ch * 64, it.h, it.q0, it.b);
        }
      }
      ++q_cnt;
      for (int jt = 0; jt < it.n_tiles; ++jt) {
        if (!wait_phase_warp(&c.st_empty[st], st_par ^ 1, wc)) { ok = false; break; }
        if (lane == 0) {
          mbar_expect_tx(&c.st_full[st], 2 * kKTile);
          for (int ch = 0; ch < kChunks; ++ch) {
            tma_load_4d(sK + st * kKTile + ch * kKChunk, &p.tm_k, &c.st_full[st], ch * 64, it.kvh, jt * kKT, it.b);
            tma_load_4d(sV + st * kKTile + ch * kKChunk, &p.tm_v, &c.st_full[st], ch * 64, it.kvh, jt * kKT, it.b);
          }
        }
        issued |= 1u << st;
        last_par = (last_par & ~(1u << st)) | (st_par << st);
        if (dq_needs_fix(jt, it.L, p.Skv)) {
          if (!wait_phase_warp(&c.st_full[st], st_par, wc)) { ok = false; break; }
          const int r0 = it.L - jt * kKT;  // >= 1: tile jt holds valid keys
          const int units = (kKT - r0) * kChunks * 8;
          uint8_t* base = sK + st * kKTile;
          for (int e = lane; e < units; e += 32) {
            const int rr = r0 + e / (kChunks * 8);
            const int rest = e % (kChunks * 8);
            *reinterpret_cast<uint4*>(base + (rest / 8) * kKChunk + rr * 128 + (rest % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&c.st_fixed[st]);
        }
        if (++st == NST) { st = 0; st_par ^= 1; }
      }
    }
    for (int s = 0; s < NST; ++s)
      if (issued & (1u << s)) wait_phase_teardown(&c.st_full[s], (last_par >> s) & 1, kTeardownNs);
    if (q_cnt > 0) wait_phase_teardown(&c.q_full, (q_cnt - 1) & 1, kTeardownNs);
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t sQa = smem_u32(sQ), sdOa = smem_u32(sdO);
      const uint32_t sKa = smem_u32(sK), sVa = smem_u32(sV);
      uint32_t q_cnt = 0, st = 0, st_par = 0, fix_par = 0, gt = 0, item_cnt = 0;
      bool ok = true;
      auto acc_mma = [&](uint32_t tg, uint32_t s, bool first) -> bool {
        const uint32_t u = tg & 1, cu = tg >> 1;
        if (!wait_phase(&c.ds_ready[u], cu & 1, wc)) return false;
        if (first && !wait_phase(&c.acc_free, (item_cnt & 1) ^ 1, wc)) return false;
        tc_fence_after();
        const uint32_t tbuf = tmem + D + u * 128;
#pragma unroll
        for (int kk = 0; kk < kKT / 16; ++kk) {
          const uint64_t bk = smem_desc_sw128(sKa + s * kKTile + kk * 16 * 128, kKChunk, 1024);
          mma_ts(tmem, tbuf + 64 + kk * 8, bk, kIdescAcc, (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(&c.mm2_done[u]);
        mma_commit(&c.st_empty[s]);
        return true;
      };
      for (int idx = blockIdx.x; ok && idx < p.n_items; idx += gridDim.x) {
        const DqItem it = dq_decode(idx, p);
        if (it.n_tiles == 0) continue;
        if (!wait_phase(&c.q_full, q_cnt & 1, wc)) { ok = false; break; }
        tc_fence_after();
        uint32_t prev_st = 0;
        for (int jt = 0; jt < it.n_tiles; ++jt) {
          const uint32_t u = gt & 1, cu = gt >> 1;
          if (dq_needs_fix(jt, it.L, p.Skv)) {
            if (!wait_phase(&c.st_fixed[st], (fix_par >> st) & 1, wc)) { ok = false; break; }
            fix_par ^= 1u << st;
          } else if (!wait_phase(&c.st_full[st], st_par, wc)) {
            ok = false;
            break;
          }
          if (cu >= 1 && !wait_phase(&c.mm2_done[u], (cu - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tbuf = tmem + D + u * 128;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk % 4) * 32;
            const uint64_t aq = smem_desc_sw128(sQa + (kk / 4) * kQChunk + off, 16, 1024);
            const uint64_t bk = smem_desc_sw128(sKa + st * kKTile + (kk / 4) * kKChunk + off, 16, 1024);
            mma_ss(tbuf, aq, bk, kIdescSP, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk % 4) * 32;
            const uint64_t ado = smem_desc_sw128(sdOa + (kk / 4) * kQChunk + off, 16, 1024);
            const uint64_t bv = smem_desc_sw128(sVa + st * kKTile + (kk / 4) * kKChunk + off, 16, 1024);
            mma_ss(tbuf + 64, ado, bv, kIdescSP, kk > 0 ? 1u : 0u);
          }
          mma_commit(&c.sp_full[u]);
          if (jt >= 1 && !acc_mma(gt - 1, prev_st, jt == 1)) { ok = false; break; }
          prev_st = st;
          if (++st == NST) { st = 0; st_par ^= 1; }
          ++gt;
        }
        if (!ok) break;
        if (!acc_mma(gt - 1, prev_st, it.n_tiles == 1)) { ok = false; break; }
        mma_commit(&c.acc_done);
        mma_commit(&c.q_empty);
        ++q_cnt;
        ++item_cnt;
      }
      mma_commit(&c.mma_final);
      wait_phase_teardown(&c.mma_final, 0, kTeardownNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- elementwise
    const int w = (warp - 2) / 4;
    const int quad = warp % 4;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t gt = 0, item_cnt = 0;
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < p.n_items; idx += gridDim.x) {
      const DqItem it = dq_decode(idx, p);
      const int i = it.q0 + r;
      const bool row_ok = i < p.Sq;
      __nv_bfloat16* dst = p.dq + ((static_cast<int64_t>(it.b) * p.Sq + i) * p.Hq + it.h) * D + w * (D / 2);
      if (it.n_tiles == 0) {
        if (row_ok) zero_row_bf16(dst, D / 2);
        continue;
      }
      const int64_t srow = (static_cast<int64_t>(it.b) * p.Hq + it.h) * p.Sq + i;
      float l2 = CUDART_INF_F, dl = 0.f;
      if (row_ok) {
        const float lv = __ldg(p.lse + srow);
        l2 = lv == -CUDART_INF_F ? CUDART_INF_F : lv * kLog2e;
        dl = __ldg(p.delta + srow);
      }
      const int kend = p.causal ? min(it.L, i + it.L - p.Sq + 1) : it.L;
      for (int jt = 0; jt < it.n_tiles; ++jt, ++gt) {
        if (static_cast<int>(gt & 1) != w) continue;
        if (!wait_phase_warp(&c.sp_full[w], (gt >> 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tbuf = tmem + lane_off + D + w * 128;
        const int limit = kend - jt * kKT;
        uint32_t dd[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float sv[32], dp[32];
          tmem_ld32(tbuf + half * 32, reinterpret_cast<uint32_t*>(sv));
          tmem_ld32(tbuf + 64 + half * 32, reinterpret_cast<uint32_t*>(dp));
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float d2[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int q = half * 32 + 2 * e + h2;
              const bool vis = q < limit;
              const float pq = vis ? ex2_approx(fmaf(sv[2 * e + h2], p.scale_log2, -l2)) : 0.f;
              d2[h2] = vis ? pq * (dp[2 * e + h2] - dl) : 0.f;
            }
            dd[half * 16 + e] = pack_bf16x2(d2[0], d2[1]);
          }
        }
        tmem_st32(tbuf + 64, dd);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&c.ds_ready[w]);
      }
      if (!ok) break;
      if (!wait_phase_warp(&c.acc_done, item_cnt & 1, wc)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + w * (D / 2) + cc * 32, v);
        if (row_ok) store_row_bf16(dst + cc * 32, v, p.scale);
      }
      tc_fence_before();
      mbar_arrive(&c.acc_free);
      ++item_cnt;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ===================================================================== group reduction
// Split mode: dK[b, j, kvh] = scale * sum over the group's query heads r = 0 .. g - 1 (in
// that order) of the partial dK[b, j, kvh * g + r]; likewise dV (unscaled). Each thread
// reduces 4 consecutive elements of one (b, j, kvh) row.
__global__ void __launch_bounds__(256) bwd_group_reduce_kernel(const float* __restrict__ part_dk,
                                                               const float* __restrict__ part_dv,
                                                               __nv_bfloat16* dk, __nv_bfloat16* dv,
                                                               int B, int Skv, int Hq, int Hkv, int D,
                                                               float scale) {
  const int g = Hq / Hkv;
  const int64_t n4 = (int64_t)B * Skv * Hkv * D / 4;
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n4) return;
  const int d4 = (int)(e % (D / 4));
  const int64_t row = e / (D / 4);  // (b * Skv + j) * Hkv + kvh
  const int kvh = (int)(row % Hkv);
  const int64_t bj = row / Hkv;
  const int64_t src0 = (bj * Hq + (int64_t)kvh * g) * D + 4 * d4;
  float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sv = sk;
  for (int r = 0; r < g; ++r) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(part_dk + src0 + (int64_t)r * D));
    const float4 c = __ldg(reinterpret_cast<const float4*>(part_dv + src0 + (int64_t)r * D));
    sk.x += a.x; sk.y += a.y; sk.z += a.z; sk.w += a.w;
    sv.x += c.x; sv.y += c.y; sv.z += c.z; sv.w += c.w;
  }
  const int64_t dst = row * D + 4 * d4;
  *reinterpret_cast<uint2*>(dk + dst) =
      make_uint2(pack_bf16x2(sk.x * scale, sk.y * scale), pack_bf16x2(sk.z * scale, sk.w * scale));
  *reinterpret_cast<uint2*>(dv + dst) = make_uint2(pack_bf16x2(sv.x, sv.y), pack_bf16x2(sv.z, sv.w));
}

// ============================================================================ host side
template <int D, int NST>
constexpr size_t dkdv_smem() {
  return 1024 + 2 * (size_t)kKeys * D * 2 + 2 * (size_t)NST * kQT * D * 2 + sizeof(DkvCtl<NST>);
}
template <int D, int NST>
constexpr size_t dq_smem() {
  return 1024 + 2 * (size_t)kQRows * D * 2 + 2 * (size_t)NST * kKT * D * 2 + sizeof(DqCtl<NST>);
}

constexpr int kMaxDev = 64;
std::mutex g_mu;
int g_num_sms[kMaxDev] = {};
bool g_attr[kMaxDev][4] = {};

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes, int dev, int which) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_attr[dev][which]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    g_attr[dev][which] = true;
  }
  return cudaSuccess;
}

template <int D>
cudaError_t launch_bwd(const Problem& p, int dev, cudaStream_t s) {
  constexpr int NST_KV = D == 64 ? 6 : 4;
  constexpr int NST_Q = D == 64 ? 6 : 4;
  BwdParams prm{};
  const bool no_keys = p.Skv == 0;
  if (!make_bshd_map(&prm.tm_q, p.q, p.B, p.Sq, p.Hq, D, kQT) ||
      !make_bshd_map(&prm.tm_do, p.dout, p.B, p.Sq, p.Hq, D, kQT) ||
      !make_bshd_map(&prm.tm_k, no_keys ? p.q : p.k, p.B, no_keys ? p.Sq : p.Skv,
                     no_keys ? p.Hq : p.Hkv, D, kKeys) ||
      !make_bshd_map(&prm.tm_v, no_keys ? p.q : p.v, p.B, no_keys ? p.Sq : p.Skv,
                     no_keys ? p.Hq : p.Hkv, D, kKeys))
    return cudaErrorInvalidValue;
  prm.lse = p.lse;
  prm.delta = p.delta;
  prm.dq = static_cast<__nv_bfloat16*>(p.dq);
  prm.dk = static_cast<__nv_bfloat16*>(p.dk);
  prm.dv = static_cast<__nv_bfloat16*>(p.dv);
  prm.part_dk = p.part_dk;
  prm.part_dv = p.part_dv;
  prm.split = p.split;
  prm.kv_lens = p.kv_lens;
  prm.err = p.err;
  prm.B = p.B;
  prm.Hq = p.Hq;
  prm.Hkv = p.Hkv;
  prm.Sq = p.Sq;
  prm.Skv = p.Skv;
  prm.causal = p.causal;
  prm.scale = p.scale;
  prm.scale_log2 = p.scale * kLog2e;
  prm.timeout_ns = 4000000000ull;
  const int sms = g_num_sms[dev];
  if (p.Skv > 0) {
    prm.n_items = p.B * p.Hkv * ((p.Skv + kKeys - 1) / kKeys) * (p.split ? p.Hq / p.Hkv : 1);
    constexpr size_t smem = dkdv_smem<D, NST_KV>();
    cudaError_t e = set_smem(bwd_dkdv_sm103_kernel<D, NST_KV>, smem, dev, D == 64 ? 0 : 1);
    if (e != cudaSuccess) return e;
    bwd_dkdv_sm103_kernel<D, NST_KV><<<prm.n_items < sms ? prm.n_items : sms, kThreads, smem, s>>>(prm);
    count_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.split) {
      const int64_t n4 = (int64_t)p.B * p.Skv * p.Hkv * D / 4;
      bwd_group_reduce_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(
          p.part_dk, p.part_dv, prm.dk, prm.dv, p.B, p.Skv, p.Hq, p.Hkv, D, p.scale);
      count_launches(1);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  // the dQ kernel tiles K/V by 64 keys and Q/dO by 128 rows
  if (!make_bshd_map(&prm.tm_q, p.q, p.B, p.Sq, p.Hq, D, kQRows) ||
      !make_bshd_map(&prm.tm_do, p.dout, p.B, p.Sq, p.Hq, D, kQRows) ||
      !make_bshd_map(&prm.tm_k, no_keys ? p.q : p.k, p.B, no_keys ? p.Sq : p.Skv,
                     no_keys ? p.Hq : p.Hkv, D, kKT) ||
      !make_bshd_map(&prm.tm_v, no_keys ? p.q : p.v, p.B, no_keys ? p.Sq : p.Skv,
                     no_keys ? p.Hq : p.Hkv, D, kKT))
    return cudaErrorInvalidValue;
  prm.n_items = p.B * p.Hq * ((p.Sq + kQRows - 1) / kQRows);
  constexpr size_t smem = dq_smem<D, NST_Q>();
  cudaError_t e = set_smem(bwd_dq_sm103_kernel<D, NST_Q>, smem, dev, D == 64 ? 2 : 3);
  if (e != cudaSuccess) return e;
  bwd_dq_sm103_kernel<D, NST_Q><<<prm.n_items < sms ? prm.n_items : sms, kThreads, smem, s>>>(prm);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc_bwd(const Problem& p, cudaStream_t s) {
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
  // delta = rowsum(dO * O) into the workspace first
  e = simt_delta(p, s);
  if (e != cudaSuccess) return e;
  return p.D == 64 ? launch_bwd<64>(p, dev, s) : launch_bwd<128>(p, dev, s);
}

}  // namespace attn
