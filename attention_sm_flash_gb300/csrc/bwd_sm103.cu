// bf16 attention backward for sm_103a: tcgen05 MMAs into TMEM, TMA-staged tiles.
//
// The flash backward of "xtrain evolution.md" (infrastructure table, row T14): the
// scores are recomputed from Q, K and the forward's LSE, and delta = rowsum(dO * O)
// simplifies the softmax Jacobian:
//     P = exp(scale * Q K^T - LSE),  dP = dO V^T,  dS = P * (dP - delta),
//     dV = P^T dO,  dK = scale * dS^T Q,  dQ = scale * dS K.
// delta comes first from a small bandwidth-bound kernel; then two tcgen05 kernels, both
// deterministic (every sum in a fixed order, no atomics), on 128 x 128 tiles so that
// every MMA is M = 128, N = 128 (or N = D):
//
// dQ: a CTA owns 128 query rows of one (batch, head) and loops over K/V tiles of 128
//   keys: S = Q K^T, dP = dO V^T, dS on the elementwise warps, dQ += dS K. S is consumed
//   into registers as soon as it lands, so the next tile's S MMA can start while dS is
//   still being formed; dP is double-buffered (dS is written over it, bf16, as the A
//   operand of dQ += dS K).
// dK/dV: a CTA owns 128 keys of one (batch, kv head) and loops over the query heads of
//   the GQA group and their query tiles of 128 rows in a fixed order, so the group sum of
//   row T15 (in-group deterministic sum) happens inside its TMEM accumulators. When such
//   items are too few to fill the GPU (few kv heads, causal imbalance), the group's
//   query heads are split into a few runs of consecutive heads, each its own item writing
//   fp32 partial dK/dV, and a reduction kernel sums each group's partials in head order -
//   still deterministic, still no atomics. Keys sit on the TMEM lanes:
//   S^T = K Q^T and dP^T = V dO^T. The elementwise warps read S^T into registers (which
//   frees its columns for the next tile's S^T), write P^T (bf16) to a shared-memory tile
//   for dV += P^T dO, and write dS^T (bf16) over the first columns of dP^T, from where
//   dK += dS^T Q takes A. The MMAs of one tile are issued S^T, dP^T, dV, dK, so that each
//   wait of the issuing threads (P^T ready, dS^T ready, S^T's columns free, dP^T's columns
//   free) sits behind an MMA already queued. A Q/dO stage is released in two halves: dO
//   once dP^T and dV have read it, Q once dK has.
//
// Roles (384 threads): warp 0 TMA producer; two MMA-issuing threads, one in warp 1 for the
// products that recompute S and dP, one in warp 10 for the accumulations (dQ, or dV and
// dK), since one thread alone spends about as long issuing a tile's MMAs as the tensor
// pipe spends executing them; warps 2-9 elementwise: warp w reaches the TMEM lanes
// 32 * (w % 4) .. and takes the 64 columns 64 * ((w - 2) / 4) .. of each 128-column tile;
// in the dQ kernel warp 11 stages the next work item's per-row LSE and delta.
// Work items are dealt to the persistent CTAs in a snake order (CTA c takes items c,
// 2G - 1 - c, 2G + c, ...), so that on longest-first item lists long and short items
// pair up. Every barrier wait is bounded in time; a wait that runs out flags
// ATTN_DEVERR_TIMEOUT and the CTA gives up after letting its copies and MMAs in flight
// finish.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <mutex>

#include "attn_internal.h"
#include "fastdiv.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

using namespace sm103;

constexpr int kThreads = 384;  // warp 0 producer, warps 1 and 10 MMA issuers, warps 2-9 elementwise
constexpr int kAccWarp = 10;
constexpr int kStatWarp = 11;   // dQ kernel: stages per-row LSE and delta, one item ahead
constexpr int kEwThreads = 256;
constexpr int kEwWarps = kEwThreads / 32;  // the count of barriers the elementwise warps arrive on
constexpr int kT = 128;        // rows of every tile: keys and queries alike
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kTeardownNs = 200000000ull;

struct BwdParams {
  CUtensorMap tm_q, tm_do, tm_k, tm_v;
  const __nv_bfloat16* o;     // the forward's O, [B, Sq, Hq, D]
  const __nv_bfloat16* dout;  // dO, same layout
  const float* lse;
  float* delta;  // rowsum(dO * O), [B, Hq, Sq], written by bwd_delta_kernel
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  // split mode: fp32 partial dK, dV [B, Skv, Hkv * split, D]; slot kvh * split + r holds
  // the sum over query heads kvh * g + r * g / split .. + g / split - 1 (g = Hq / Hkv)
  float* part_dk;
  float* part_dv;
  const int32_t* kv_lens;
  unsigned int* err;
  int B, Hq, Hkv, Sq, Skv, causal;
  int split;  // parts per GQA group (0: not split)
  int n_items;
  // the divisions of the work decode, as multiplies (fastdiv.h): dQ items by B * Hq, Hq,
  // the query tiles n_qt and the group g = Hq / Hkv; dK/dV items by B * Hkv * gs, n_kt * gs,
  // gs (items per (batch, kv head, key tile)) and Hkv
  FastDiv fd_bh, fd_hq, fd_nqt, fd_g, fd_bkgs, fd_ktgs, fd_gs, fd_hkv;
  int heads_per_item;  // g / gs
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

// the same with 32-byte stores (dst 32-byte aligned): half the store instructions, and a
// warp's store touches 32 rows either way
__device__ __forceinline__ void store_row_bf16_v8(__nv_bfloat16* dst, const uint32_t* v, float mul) {
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e)
    pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
  st_global_v8(dst, pk);
  st_global_v8(dst + 16, pk + 8);
}

__device__ __forceinline__ void zero_row_bf16(__nv_bfloat16* dst, int n) {
  for (int d = 0; d < n; d += 8) *reinterpret_cast<uint4*>(dst + d) = make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ int item_at(int pass) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return (pass & 1) ? (pass + 1) * G - 1 - c : pass * G + c;
}

// Loads that the SW128 K-major / MN-major descriptors below address: a tile of `rows`
// rows and D columns is D / 64 chunks of rows x 128 bytes (8-row groups 1024 bytes apart).
template <int D>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int head,
                                          int row0, int b, int rows) {
#pragma unroll
  for (int ch = 0; ch < D / 64; ++ch) tma_load_4d(dst + ch * rows * 128, map, bar, ch * 64, head, row0, b);
}

// =============================================================================== dQ
// K and V ride separate rings: V(g) is free once dP(g) completes, K(g) only after
// dQ(g) += dS(g) K(g), which comes a tile later; so K gets the deeper ring.
template <int NK, int NV>
struct DqCtl {
  uint64_t q_full, q_empty, do_full, do_empty;
  uint64_t k_full[NK], k_empty[NK], k_fixed[NK];
  uint64_t v_full[NV], v_empty[NV];
  uint64_t s_full, s_free;
  uint64_t dp_full[2], ds_ready[2], dq_done[2];
  uint64_t acc_done, acc_free, mma_final, mma_final2;
  uint64_t dl_full, dl_free;
  uint32_t tmem_base;
  int abort;
  float nlse[kT];   // -LSE * log2(e) and delta of the rows of the next item with tiles
  float delta[kT];
};

struct DqItem {
  int b, h, kvh, q0, L, n_tiles;
};

__device__ __forceinline__ DqItem dq_decode(int idx, const BwdParams& p) {
  const int n_qt = p.fd_nqt.d;
  int b, h, qt;
  if (p.causal) {
    const int r = p.fd_bh.div(idx);
    qt = n_qt - 1 - r;  // longest first
    const int bh = idx - r * p.fd_bh.d;
    b = p.fd_hq.div(bh);
    h = bh - b * p.Hq;
  } else {
    const int bh = p.fd_nqt.div(idx);
    qt = idx - bh * n_qt;
    b = p.fd_hq.div(bh);
    h = bh - b * p.Hq;
  }
  DqItem it;
  it.b = b;
  it.h = h;
  it.kvh = p.fd_g.div(h);
  it.q0 = qt * kT;
  it.L = kv_len_of(p, b, it.kvh);
  int kmax = it.L;
  if (p.causal) {
    const int ilast = min(it.q0 + kT - 1, p.Sq - 1);
    kmax = min(it.L, ilast + it.L - p.Sq + 1);
  }
  kmax = max(kmax, 0);
  it.n_tiles = (kmax + kT - 1) / kT;
  return it;
}

// K tile j holds in-bounds rows at or past the valid length (padding, maybe NaN); they
// are zeroed before dQ += dS K reads them.
__device__ __forceinline__ bool dq_needs_fix(int j, int L, int Skv) {
  return min(Skv, (j + 1) * kT) > L;
}

template <int D, int NK, int NV>
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_sm103_kernel(const __grid_constant__ BwdParams p) {
  constexpr int kTile = kT * D * 2;  // bytes of one Q, dO, K or V tile
  constexpr int kChunk = kT * 128;
  constexpr int kChunks = D / 64;
  constexpr uint32_t kIdescSP = idesc_bf16_f32(kT, kT, false, false);
  constexpr uint32_t kIdescAcc = idesc_bf16_f32(kT, D, false, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sdO = smem + kTile;
  uint8_t* sK = smem + 2 * kTile;              // NK stages
  uint8_t* sV = smem + (2 + NK) * kTile;       // NV stages
  DqCtl<NK, NV>& c = *reinterpret_cast<DqCtl<NK, NV>*>(smem + (2 + NK + NV) * kTile);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // the dK/dV kernel that follows reads none of this kernel's output: it may take each SM
  // as soon as this kernel's CTA there exits
  griddep_launch_dependents();

  if (threadIdx.x == 0) {
    mbar_init(&c.q_full, 1);
    mbar_init(&c.q_empty, 1);
    mbar_init(&c.do_full, 1);
    mbar_init(&c.do_empty, 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(&c.k_full[s], 1);
      mbar_init(&c.k_empty[s], 1);
      mbar_init(&c.k_fixed[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&c.v_full[s], 1);
      mbar_init(&c.v_empty[s], 1);
    }
    mbar_init(&c.s_full, 1);
    mbar_init(&c.s_free, kEwWarps);
    for (int u = 0; u < 2; ++u) {
      mbar_init(&c.dp_full[u], 1);
      mbar_init(&c.ds_ready[u], kEwWarps);
      mbar_init(&c.dq_done[u], 1);
    }
    mbar_init(&c.acc_done, 1);
    mbar_init(&c.acc_free, kEwWarps);
    mbar_init(&c.mma_final, 1);
    mbar_init(&c.mma_final2, 1);
    mbar_init(&c.dl_full, 1);
    mbar_init(&c.dl_free, kEwWarps);
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
  // TMEM columns: S [0, 128), dP double buffer [128, 384), dQ [384, 384 + D)
  const uint32_t tmem = c.tmem_base;
  const uint32_t t_s = tmem, t_dp0 = tmem + 128, t_dq = tmem + 384;
  WaitCtl wc{&c.abort, p.err, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    uint32_t q_cnt = 0, do_cnt = 0, kpos = 0, vpos = 0, k_iss = 0, k_last = 0, v_iss = 0, v_last = 0;
    bool ok = true;
    for (int ps = 0, idx = item_at(0); ok && idx < p.n_items; idx = item_at(++ps)) {
      const DqItem it = dq_decode(idx, p);
      if (it.n_tiles == 0) continue;
      if (!wait_phase_warp(&c.q_empty, (q_cnt & 1) ^ 1, wc)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(&c.q_full, kTile);
        load_tile<D>(sQ, &p.tm_q, &c.q_full, it.h, it.q0, it.b, kT);
      }
      ++q_cnt;
      if (!wait_phase_warp(&c.do_empty, (do_cnt & 1) ^ 1, wc)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(&c.do_full, kTile);
        load_tile<D>(sdO, &p.tm_do, &c.do_full, it.h, it.q0, it.b, kT);
      }
      ++do_cnt;
      for (int jt = 0; jt < it.n_tiles; ++jt, ++kpos, ++vpos) {
        const uint32_t ks = kpos % NK, kpar = (kpos / NK) & 1;
        const uint32_t vs = vpos % NV, vpar = (vpos / NV) & 1;
        if (!wait_phase_warp(&c.k_empty[ks], kpar ^ 1, wc)) { ok = false; break; }
        if (lane == 0) {
          mbar_expect_tx(&c.k_full[ks], kTile);
          load_tile<D>(sK + ks * kTile, &p.tm_k, &c.k_full[ks], it.kvh, jt * kT, it.b, kT);
        }
        k_iss |= 1u << ks;
        k_last = (k_last & ~(1u << ks)) | (kpar << ks);
        if (!wait_phase_warp(&c.v_empty[vs], vpar ^ 1, wc)) { ok = false; break; }
        if (lane == 0) {
          mbar_expect_tx(&c.v_full[vs], kTile);
          load_tile<D>(sV + vs * kTile, &p.tm_v, &c.v_full[vs], it.kvh, jt * kT, it.b, kT);
        }
        v_iss |= 1u << vs;
        v_last = (v_last & ~(1u << vs)) | (vpar << vs);
        if (dq_needs_fix(jt, it.L, p.Skv)) {
          if (!wait_phase_warp(&c.k_full[ks], kpar, wc)) { ok = false; break; }
          const int r0 = it.L - jt * kT;  // >= 1: tile jt holds valid keys
          const int units = (kT - r0) * kChunks * 8;
          uint8_t* base = sK + ks * kTile;
          for (int e = lane; e < units; e += 32) {
            const int rr = r0 + e / (kChunks * 8);
            const int rest = e % (kChunks * 8);
            *reinterpret_cast<uint4*>(base + (rest / 8) * kChunk + rr * 128 + (rest % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&c.k_fixed[ks]);
        }
      }
    }
    // every copy this CTA started lands before its shared memory can go away
    for (int s = 0; s < NK; ++s)
      if (k_iss & (1u << s)) wait_phase_teardown(&c.k_full[s], (k_last >> s) & 1, kTeardownNs);
    for (int s = 0; s < NV; ++s)
      if (v_iss & (1u << s)) wait_phase_teardown(&c.v_full[s], (v_last >> s) & 1, kTeardownNs);
    if (q_cnt > 0) wait_phase_teardown(&c.q_full, (q_cnt - 1) & 1, kTeardownNs);
    if (do_cnt > 0) wait_phase_teardown(&c.do_full, (do_cnt - 1) & 1, kTeardownNs);
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer: S and dP
    // S(g) waits until S(g - 1) has been read into registers, dP(g) until dQ(g - 2) has
    // read dS(g - 2) (same buffer)
    if (lane == 0) {
      const uint32_t sQa = smem_u32(sQ), sdOa = smem_u32(sdO);
      const uint32_t sKa = smem_u32(sK), sVa = smem_u32(sV);
      uint32_t q_cnt = 0, fix_par = 0, gt = 0;
      bool ok = true;
      for (int ps = 0, idx = item_at(0); ok && idx < p.n_items; idx = item_at(++ps)) {
        const DqItem it = dq_decode(idx, p);
        if (it.n_tiles == 0) continue;
        for (int jt = 0; jt < it.n_tiles; ++jt, ++gt) {
          const uint32_t u = gt & 1;
          const uint32_t ks = gt % NK, vs = gt % NV;
          if (dq_needs_fix(jt, it.L, p.Skv)) {
            if (!wait_phase(&c.k_fixed[ks], (fix_par >> ks) & 1, wc)) { ok = false; break; }
            fix_par ^= 1u << ks;
          } else if (!wait_phase(&c.k_full[ks], (gt / NK) & 1, wc)) {
            ok = false;
            break;
          }
          if (jt == 0 && !wait_phase(&c.q_full, q_cnt & 1, wc)) { ok = false; break; }
          if (gt >= 1 && !wait_phase(&c.s_free, (gt - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * kChunk + (kk % 4) * 32;
            mma_ss(t_s, smem_desc_sw128(sQa + off, 16, 1024), smem_desc_sw128(sKa + ks * kTile + off, 16, 1024),
                   kIdescSP, kk > 0 ? 1u : 0u);
          }
          mma_commit(&c.s_full);
          if (jt == it.n_tiles - 1) mma_commit(&c.q_empty);
          if (!wait_phase(&c.v_full[vs], (gt / NV) & 1, wc)) { ok = false; break; }
          if (jt == 0 && !wait_phase(&c.do_full, q_cnt & 1, wc)) { ok = false; break; }
          if (gt >= 2 && !wait_phase(&c.dq_done[u], ((gt >> 1) - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * kChunk + (kk % 4) * 32;
            mma_ss(t_dp0 + u * 128, smem_desc_sw128(sdOa + off, 16, 1024),
                   smem_desc_sw128(sVa + vs * kTile + off, 16, 1024), kIdescSP, kk > 0 ? 1u : 0u);
          }
          mma_commit(&c.dp_full[u]);
          mma_commit(&c.v_empty[vs]);
          if (jt == it.n_tiles - 1) mma_commit(&c.do_empty);
        }
        ++q_cnt;
      }
      mma_commit(&c.mma_final);
      wait_phase_teardown(&c.mma_final, 0, kTeardownNs);
    }
    __syncwarp();
  } else if (warp == kAccWarp) {
    // --------------------------------------------------- MMA issuer: dQ += dS K
    // dS(g) ready implies S(g) complete, so the commit to K's empty barrier also covers
    // the other issuer's read of K(g)
    if (lane == 0) {
      const uint32_t sKa = smem_u32(sK);
      uint32_t gt = 0, item_cnt = 0;
      bool ok = true;
      for (int ps = 0, idx = item_at(0); ok && idx < p.n_items; idx = item_at(++ps)) {
        const DqItem it = dq_decode(idx, p);
        if (it.n_tiles == 0) continue;
        for (int jt = 0; jt < it.n_tiles; ++jt, ++gt) {
          const uint32_t u = gt & 1, ks = gt % NK;
          if (!wait_phase(&c.ds_ready[u], (gt >> 1) & 1, wc)) { ok = false; break; }
          if (jt == 0 && !wait_phase(&c.acc_free, (item_cnt & 1) ^ 1, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = t_dp0 + u * 128;
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk) {
            // dS columns: keys 64 h .. 64 h + 63 were written at 64 h .. 64 h + 31
            const uint64_t bk = smem_desc_sw128(sKa + ks * kTile + kk * 16 * 128, kChunk, 1024);
            mma_ts(t_dq, a0 + (kk / 4) * 64 + (kk % 4) * 8, bk, kIdescAcc, (jt == 0 && kk == 0) ? 0u : 1u);
          }
          mma_commit(&c.dq_done[u]);
          mma_commit(&c.k_empty[ks]);
        }
        if (!ok) break;
        mma_commit(&c.acc_done);
        ++item_cnt;
      }
      mma_commit(&c.mma_final2);
      wait_phase_teardown(&c.mma_final2, 0, kTeardownNs);
    }
    __syncwarp();
  } else if (warp == kStatWarp) {
    // ------------------------------------------- per-row LSE and delta, one item ahead
    // stages -LSE * log2(e) (-inf: the row sees no key or is past the end) and delta of
    // the item's 128 rows in shared memory, so the elementwise warps start an item
    // without a global load
    uint32_t dcnt = 0;
    bool ok = true;
    for (int ps = 0, idx = item_at(0); ok && idx < p.n_items; idx = item_at(++ps)) {
      const DqItem it = dq_decode(idx, p);
      if (it.n_tiles == 0) continue;
      // the elementwise warps read the previous item's values as they start it
      if (dcnt >= 1 && !wait_phase_warp(&c.dl_free, (dcnt - 1) & 1, wc)) { ok = false; break; }
      const int64_t srow0 = (static_cast<int64_t>(it.b) * p.Hq + it.h) * p.Sq + it.q0;
#pragma unroll
      for (int k2 = 0; k2 < kT / 32; ++k2) {
        const int rr = lane + 32 * k2;
        float nl2 = -CUDART_INF_F, dl = 0.f;
        if (it.q0 + rr < p.Sq) {
          const float lv = __ldg(p.lse + srow0 + rr);
          nl2 = lv == -CUDART_INF_F ? -CUDART_INF_F : -lv * kLog2e;
          dl = p.delta[srow0 + rr];
        }
        c.nlse[rr] = nl2;
        c.delta[rr] = dl;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.dl_full);
      ++dcnt;
    }
  } else if (warp < kAccWarp) {
    // ------------------------------------------------------------- elementwise
    const int hsel = (warp - 2) / 4;  // columns 64 hsel .. 64 hsel + 63 of each tile
    const int quad = warp % 4;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    // dQ rows start 32-byte aligned when the tensor does (row and column offsets are
    // multiples of 64 bytes)
    const bool out32 = (reinterpret_cast<uintptr_t>(p.dq) & 31u) == 0u;
    uint32_t gt = 0, item_cnt = 0, dcnt = 0;
    bool ok = true;
    for (int ps = 0, idx = item_at(0); ok && idx < p.n_items; idx = item_at(++ps)) {
      const DqItem it = dq_decode(idx, p);
      const int i = it.q0 + r;
      const bool row_ok = i < p.Sq;
      const int64_t qrow = (static_cast<int64_t>(it.b) * p.Sq + i) * p.Hq + it.h;
      __nv_bfloat16* dst = p.dq + qrow * D + hsel * (D / 2);
      if (it.n_tiles == 0) {
        if (row_ok) zero_row_bf16(dst, D / 2);
        continue;
      }
      // this row's LSE and delta, staged by warp 11; a row that sees no key (LSE = -inf)
      // and a row past the end get P = 0
      if (!wait_phase_warp(&c.dl_full, dcnt & 1, wc)) { ok = false; break; }
      const float dl = c.delta[r], nl2 = c.nlse[r];
      mbar_arrive_warp(&c.dl_free);
      ++dcnt;
      const float2 nl2v = make_float2(nl2, nl2), ndl = make_float2(-dl, -dl);
      // keys j < kend are visible to this row
      const int kend = p.causal ? min(it.L, i + it.L - p.Sq + 1) : it.L;
      for (int jt = 0; jt < it.n_tiles; ++jt, ++gt) {
        const uint32_t u = gt & 1;
        if (!wait_phase_warp(&c.s_full, gt & 1, wc)) { ok = false; break; }
        tc_fence_after();
        float pr[64];
        tmem_ld64(t_s + lane_off + 64 * hsel, reinterpret_cast<uint32_t*>(pr));
        tc_fence_before();
        mbar_arrive_warp(&c.s_free);
        const int limit = kend - jt * kT - 64 * hsel;
        // every key of this half visible to every row of the warp: no masking
        const bool full = __all_sync(0xffffffffu, limit >= 64);
        if (full) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float2 x = f2fma(make_float2(pr[2 * e], pr[2 * e + 1]), sl2, nl2v);
            pr[2 * e] = ex2_approx(x.x);
            pr[2 * e + 1] = ex2_approx(x.y);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) pr[e] = e < limit ? ex2_approx(fmaf(pr[e], p.scale_log2, nl2)) : 0.f;
        }
        if (!wait_phase_warp(&c.dp_full[u], (gt >> 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tdp = t_dp0 + u * 128 + lane_off + 64 * hsel;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float dp[32];
          tmem_ld32(tdp + 32 * half, reinterpret_cast<uint32_t*>(dp));
          uint32_t dd[16];
          if (full) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int c0 = 32 * half + 2 * e;
              const float2 d = f2mul(f2add(make_float2(dp[2 * e], dp[2 * e + 1]), ndl),
                                     make_float2(pr[c0], pr[c0 + 1]));
              dd[e] = pack_bf16x2(d.x, d.y);
            }
          } else {
            // a masked key may hold padding (NaN) in dP: select, not multiply by P = 0
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int c0 = 32 * half + 2 * e;
              const float d0 = c0 < limit ? pr[c0] * (dp[2 * e] - dl) : 0.f;
              const float d1 = c0 + 1 < limit ? pr[c0 + 1] * (dp[2 * e + 1] - dl) : 0.f;
              dd[e] = pack_bf16x2(d0, d1);
            }
          }
          tmem_st16(tdp + 16 * half, dd);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(&c.ds_ready[u]);
      }
      if (!ok) break;
      if (!wait_phase_warp(&c.acc_done, item_cnt & 1, wc)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t v[32];
        tmem_ld32(t_dq + lane_off + hsel * (D / 2) + cc * 32, v);
        if (row_ok) {
          if (out32) store_row_bf16_v8(dst + cc * 32, v, p.scale);
          else store_row_bf16(dst + cc * 32, v, p.scale);
        }
      }
      tc_fence_before();
      mbar_arrive_warp(&c.acc_free);
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

// =============================================================================== dK/dV
template <int NST>
struct DkvCtl {
  uint64_t k_full, k_empty, v_full, v_empty;
  // a stage's Q and dO are released separately: dO once dP^T and dV have read it (two
  // commits, one per issuer), Q once dK has, later in the tile
  uint64_t q_full[NST], q_empty[NST], do_full[NST], do_empty[NST];
  uint64_t s_full, s_free, p_ready, dv_done;
  // per dP^T buffer: dP^T landed / dK has read the dS^T written there. With two buffers
  // dP^T may run two tiles ahead of the elementwise warps, and a parity wait only tells
  // apart phases one apart, so each buffer has its own barrier.
  uint64_t dp_full[2], ds_ready[2], dk_done[2];
  uint64_t acc_done, acc_free, mma_final, mma_final2;
  uint32_t tmem_base;
  int abort;
  // -LSE * log2(e) of the tile's queries (-inf: the query contributes nothing), -delta
  alignas(16) float nlse[NST][kT];
  alignas(16) float ndel[NST][kT];
};

struct DkvItem {
  int b, kvh, j0, L;
  int h0, heads;  // query heads h0 .. h0 + heads - 1 (the whole group, or a run of it)
  int slot;       // split mode: the partial dK/dV slot, kvh * split + r
  int i_start, per_head, n_tiles;
};

__device__ __forceinline__ DkvItem dkv_decode(int idx, const BwdParams& p) {
  const int g = p.fd_g.d;
  const int gs = p.fd_gs.d;  // items per (batch, kv head, key tile)
  int b, kvh, kt, r;
  if (p.causal) {
    // longest first: the first key tiles are seen by the most queries
    kt = p.fd_bkgs.div(idx);
    const int rem = idx - kt * p.fd_bkgs.d;
    const int bk = p.fd_gs.div(rem);
    r = rem - bk * gs;
    b = p.fd_hkv.div(bk);
    kvh = bk - b * p.Hkv;
  } else {
    const int bk = p.fd_ktgs.div(idx);
    const int rem = idx - bk * p.fd_ktgs.d;
    kt = p.fd_gs.div(rem);
    r = rem - kt * gs;
    b = p.fd_hkv.div(bk);
    kvh = bk - b * p.Hkv;
  }
  DkvItem it;
  it.b = b;
  it.kvh = kvh;
  it.j0 = kt * kT;
  it.L = kv_len_of(p, b, kvh);
  it.heads = p.heads_per_item;
  it.h0 = kvh * g + r * it.heads;
  it.slot = kvh * gs + r;
  const int n_qt = (p.Sq + kT - 1) / kT;
  it.i_start = 0;
  it.per_head = 0;
  if (it.j0 < it.L) {
    // queries that see key j0: i >= j0 - L + Sq (causal, bottom-right)
    const int first = p.causal ? max(0, it.j0 - it.L + p.Sq) : 0;
    it.i_start = first / kT;
    it.per_head = max(0, n_qt - it.i_start);
  }
  it.n_tiles = it.heads * it.per_head;
  return it;
}

template <int D, int NST>
__global__ void __launch_bounds__(kThreads, 1) bwd_dkdv_sm103_kernel(const __grid_constant__ BwdParams p) {
  constexpr int kTile = kT * D * 2;
  constexpr int kChunk = kT * 128;
  constexpr uint32_t kIdescSP = idesc_bf16_f32(kT, kT, false, false);
  constexpr uint32_t kIdescAcc = idesc_bf16_f32(kT, D, false, true);

  // no alignment slack: every byte of the 227 KB is used, and the dynamic shared memory
  // of a kernel without static shared memory starts 1024-byte aligned (checked: the
  // 128-byte swizzle of the tiles needs it)
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicOr(p.err, ATTN_DEVERR_LAYOUT);
    // like every other exit, only after the dQ grid has completed (see the end)
    griddep_wait();
    return;
  }
  uint8_t* sK = smem;
  uint8_t* sV = smem + kTile;
  uint8_t* sQ = smem + 2 * kTile;                 // NST stages
  uint8_t* sdO = smem + 2 * kTile + NST * kTile;  // NST stages
  uint8_t* sP = smem + 2 * kTile + 2 * NST * kTile;  // P^T (bf16, keys x queries, K-major)
  DkvCtl<NST>& c = *reinterpret_cast<DkvCtl<NST>*>(sP + kT * kT * 2);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // split mode: the group reduction that follows is a programmatic dependent of this grid
  // (it waits for this grid's completion before reading the partials), so it may be
  // scheduled on the SMs this grid's CTAs leave
  if (p.split) griddep_launch_dependents();

  if (threadIdx.x == 0) {
    mbar_init(&c.k_full, 1);
    mbar_init(&c.k_empty, 1);
    mbar_init(&c.v_full, 1);
    mbar_init(&c.v_empty, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&c.q_full[s], 2);  // TMA (expect_tx) + LSE/delta stores
      mbar_init(&c.q_empty[s], 1);
      mbar_init(&c.do_full[s], 1);
      mbar_init(&c.do_empty[s], 2);
    }
    mbar_init(&c.s_full, 1);
    mbar_init(&c.s_free, kEwWarps);
    mbar_init(&c.dp_full[0], 1);
    mbar_init(&c.dp_full[1], 1);
    mbar_init(&c.p_ready, kEwWarps);
    mbar_init(&c.ds_ready[0], kEwWarps);
    mbar_init(&c.ds_ready[1], kEwWarps);
    mbar_init(&c.dv_done, 1);
    mbar_init(&c.dk_done[0], 1);
    mbar_init(&c.dk_done[1], 1);
    mbar_init(&c.acc_done, 1);
    mbar_init(&c.acc_free, kEwWarps);
    mbar_init(&c.mma_final, 1);
    mbar_init(&c.mma_final2, 1);
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
  // TMEM columns: S^T [0, 128), dP^T [128, 256), dV [256, 256 + D), dK [256 + D, 256 + 2 D).
  // P^T goes to shared memory (dV += P^T dO reads both operands there), so S^T(g + 1) may
  // be issued as soon as the elementwise warps hold S^T(g) in registers.
  const uint32_t tmem = c.tmem_base;
  // With D = 64 there is room for a second dP^T buffer [256, 384) (dV and dK move up):
  // dP^T(g + 1) then need not wait for dK(g) to read dS^T(g), which breaks the chain
  // dK(g) -> dP^T(g + 1) -> dS^T(g + 1) -> dK(g + 1) that sets the tile period.
  constexpr int NDP = D == 64 ? 2 : 1;
  const uint32_t t_s = tmem, t_dp = tmem + 128, t_dv = tmem + 128 + 128 * NDP, t_dk = t_dv + D;
  WaitCtl wc{&c.abort, p.err, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    uint32_t k_cnt = 0, v_cnt = 0, st = 0, st_par = 0, issued = 0, last_par = 0;
    bool ok = true;
    for (int ps = 0, idx = item_at(0); ok && idx < p.n_items; idx = item_at(++ps)) {
      const DkvItem it = dkv_decode(idx, p);
      if (it.n_tiles == 0) continue;
      if (!wait_phase_warp(&c.k_empty, (k_cnt & 1) ^ 1, wc)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(&c.k_full, kTile);
        load_tile<D>(sK, &p.tm_k, &c.k_full, it.kvh, it.j0, it.b, kT);
      }
      ++k_cnt;
      if (!wait_phase_warp(&c.v_empty, (v_cnt & 1) ^ 1, wc)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(&c.v_full, kTile);
        load_tile<D>(sV, &p.tm_v, &c.v_full, it.kvh, it.j0, it.b, kT);
      }
      ++v_cnt;
      // tile t is query tile it.i_start + qi of query head it.h0 + hh, kept as running
      // counters: a division by the per-item per_head would go through the MUFU
      // reciprocal, which the exponentials of the elementwise warps keep busy
      int hh = 0, qi = -1;
      for (int t = 0; t < it.n_tiles; ++t) {
        if (++qi == it.per_head) {
          qi = 0;
          ++hh;
        }
        const int h = it.h0 + hh;
        const int i0 = (it.i_start + qi) * kT;
        // dO first: its stage slot is released earlier in the tile than Q's
        if (!wait_phase_warp(&c.do_empty[st], st_par ^ 1, wc)) { ok = false; break; }
        if (lane == 0) {
          mbar_expect_tx(&c.do_full[st], kTile);
          load_tile<D>(sdO + st * kTile, &p.tm_do, &c.do_full[st], h, i0, it.b, kT);
        }
        if (!wait_phase_warp(&c.q_empty[st], st_par ^ 1, wc)) { ok = false; break; }
        if (lane == 0) {
          mbar_expect_tx(&c.q_full[st], kTile);
          load_tile<D>(sQ + st * kTile, &p.tm_q, &c.q_full[st], h, i0, it.b, kT);
        }
        issued |= 1u << st;
        last_par = (last_par & ~(1u << st)) | (st_par << st);
        const int64_t row0 = (static_cast<int64_t>(it.b) * p.Hq + h) * p.Sq;
#pragma unroll
        for (int k2 = 0; k2 < kT / 32; ++k2) {
          const int q = lane + 32 * k2;
          const int i = i0 + q;
          float nl2 = -CUDART_INF_F, nd = 0.f;
          if (i < p.Sq) {
            const float lv = __ldg(p.lse + row0 + i);
            // a row with no visible key (LSE = -inf) contributes nothing
            nl2 = lv == -CUDART_INF_F ? -CUDART_INF_F : -lv * kLog2e;
            nd = -p.delta[row0 + i];
          }
          c.nlse[st][q] = nl2;
          c.ndel[st][q] = nd;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.q_full[st]);
        if (++st == NST) { st = 0; st_par ^= 1; }
      }
    }
    for (int s = 0; s < NST; ++s)
      if (issued & (1u << s)) {
        wait_phase_teardown(&c.q_full[s], (last_par >> s) & 1, kTeardownNs);
        wait_phase_teardown(&c.do_full[s], (last_par >> s) & 1, kTeardownNs);
      }
    if (k_cnt > 0) wait_phase_teardown(&c.k_full, (k_cnt - 1) & 1, kTeardownNs);
    if (v_cnt > 0) wait_phase_teardown(&c.v_full, (v_cnt - 1) & 1, kTeardownNs);
  } else if (warp == 1) {
    // --------------------------------------------------- MMA issuer: S^T and dP^T
    // S^T(g) waits until the elementwise warps have loaded S^T(g - 1), dP^T(g) until
    // dK(g - 1) has read dS^T(g - 1) from the same columns
    if (lane == 0) {
      const uint32_t sKa = smem_u32(sK), sVa = smem_u32(sV);
      const uint32_t sQa = smem_u32(sQ), sdOa = smem_u32(sdO);
      uint32_t kv_cnt = 0, st = 0, st_par = 0, gt = 0;
      bool ok = true;
      for (int ps = 0, idx = item_at(0); ok && idx < p.n_items; idx = item_at(++ps)) {
        const DkvItem it = dkv_decode(idx, p);
        if (it.n_tiles == 0) continue;
        for (int t = 0; t < it.n_tiles; ++t) {
          if (!wait_phase(&c.q_full[st], st_par, wc)) { ok = false; break; }
          if (t == 0 && !wait_phase(&c.k_full, kv_cnt & 1, wc)) { ok = false; break; }
          if (gt >= 1 && !wait_phase(&c.s_free, (gt - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * kChunk + (kk % 4) * 32;
            mma_ss(t_s, smem_desc_sw128(sKa + off, 16, 1024), smem_desc_sw128(sQa + st * kTile + off, 16, 1024),
                   kIdescSP, kk > 0 ? 1u : 0u);
          }
          mma_commit(&c.s_full);
          if (t == it.n_tiles - 1) mma_commit(&c.k_empty);
          if (t == 0 && !wait_phase(&c.v_full, kv_cnt & 1, wc)) { ok = false; break; }
          if (!wait_phase(&c.do_full[st], st_par, wc)) { ok = false; break; }
          // dP^T(g) goes to buffer g % NDP once dK(g - NDP) has read dS^T(g - NDP) there
          const uint32_t u = gt % NDP;
          if (gt >= NDP && !wait_phase(&c.dk_done[u], ((gt / NDP) - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * kChunk + (kk % 4) * 32;
            mma_ss(t_dp + u * 128, smem_desc_sw128(sVa + off, 16, 1024), smem_desc_sw128(sdOa + st * kTile + off, 16, 1024),
                   kIdescSP, kk > 0 ? 1u : 0u);
          }
          mma_commit(&c.dp_full[u]);
          mma_commit(&c.do_empty[st]);
          if (t == it.n_tiles - 1) mma_commit(&c.v_empty);
          if (++st == NST) { st = 0; st_par ^= 1; }
          ++gt;
        }
        ++kv_cnt;
      }
      mma_commit(&c.mma_final);
      wait_phase_teardown(&c.mma_final, 0, kTeardownNs);
    }
    __syncwarp();
  } else if (warp == kAccWarp) {
    // ------------------------------------- MMA issuer: dV += P^T dO, dK += dS^T Q
    // dS^T(g) ready implies S^T(g) and dP^T(g) complete, so the commit to Q's empty
    // barrier after dK(g) also covers the other issuer's read of Q(g); dO's empty barrier
    // takes a commit from each issuer, since dP^T(g) may still run when dV(g) is issued
    if (lane == 0) {
      const uint32_t sQa = smem_u32(sQ), sdOa = smem_u32(sdO), sPa = smem_u32(sP);
      uint32_t st = 0, gt = 0, item_cnt = 0;
      bool ok = true;
      for (int ps = 0, idx = item_at(0); ok && idx < p.n_items; idx = item_at(++ps)) {
        const DkvItem it = dkv_decode(idx, p);
        if (it.n_tiles == 0) continue;
        for (int t = 0; t < it.n_tiles; ++t) {
          // dV += P^T dO, both operands in shared memory
          if (!wait_phase(&c.p_ready, gt & 1, wc)) { ok = false; break; }
          if (t == 0 && !wait_phase(&c.acc_free, (item_cnt & 1) ^ 1, wc)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk) {
            const uint32_t off = (kk / 4) * kChunk + (kk % 4) * 32;
            const uint64_t bdo = smem_desc_sw128(sdOa + st * kTile + kk * 16 * 128, kChunk, 1024);
            mma_ss(t_dv, smem_desc_sw128(sPa + off, 16, 1024), bdo, kIdescAcc, (t > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&c.dv_done);
          mma_commit(&c.do_empty[st]);
          // dK += dS^T Q
          if (!wait_phase(&c.ds_ready[gt % NDP], (gt / NDP) & 1, wc)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk) {
            const uint64_t bq = smem_desc_sw128(sQa + st * kTile + kk * 16 * 128, kChunk, 1024);
            mma_ts(t_dk, t_dp + (gt % NDP) * 128 + (kk / 4) * 64 + (kk % 4) * 8, bq, kIdescAcc, (t > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&c.dk_done[gt % NDP]);
          mma_commit(&c.q_empty[st]);
          if (++st == NST) st = 0;
          ++gt;
        }
        if (!ok) break;
        mma_commit(&c.acc_done);
        ++item_cnt;
      }
      mma_commit(&c.mma_final2);
      wait_phase_teardown(&c.mma_final2, 0, kTeardownNs);
    }
    __syncwarp();
  } else if (warp < kAccWarp) {
    // ------------------------------------------------------------- elementwise
    const int hsel = (warp - 2) / 4;  // query columns 64 hsel .. 64 hsel + 63 of each tile
    const int quad = warp % 4;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    const bool out32 = ((reinterpret_cast<uintptr_t>(p.dk) | reinterpret_cast<uintptr_t>(p.dv)) & 31u) == 0u;
    uint32_t gt = 0, item_cnt = 0;
    bool ok = true;
    for (int ps = 0, idx = item_at(0); ok && idx < p.n_items; idx = item_at(++ps)) {
      const DkvItem it = dkv_decode(idx, p);
      const int j = it.j0 + r;
      const bool key_ok = j < it.L;
      const int64_t orow = ((static_cast<int64_t>(it.b) * p.Skv + j) * p.Hkv + it.kvh) * D;
      const int64_t prow = ((static_cast<int64_t>(it.b) * p.Skv + j) * p.Hkv * p.split + it.slot) * D;
      if (it.n_tiles == 0) {
        if (j < p.Skv) {
          if (p.split) {
            float4* z = reinterpret_cast<float4*>((hsel == 0 ? p.part_dv : p.part_dk) + prow);
            for (int d = 0; d < D / 4; ++d) z[d] = make_float4(0.f, 0.f, 0.f, 0.f);
          } else {
            zero_row_bf16((hsel == 0 ? p.dv : p.dk) + orow, D);
          }
        }
        continue;
      }
      int qi = -1;  // query tile of tile t within its head (a running counter, no division)
      for (int t = 0; t < it.n_tiles; ++t, ++gt) {
        if (++qi == it.per_head) qi = 0;
        const uint32_t s = gt % NST;
        if (!wait_phase_warp(&c.q_full[s], (gt / NST) & 1, wc)) { ok = false; break; }
        // the tile's per-column -LSE go to registers before the wait for S^T: while SS MMAs
        // run they take the whole shared-memory bandwidth, and a load issued on the
        // critical path costs several hundred cycles
        float4 nlv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) nlv[e] = reinterpret_cast<const float4*>(&c.nlse[s][64 * hsel])[e];
        if (!wait_phase_warp(&c.s_full, gt & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const int i0 = (it.i_start + qi) * kT + 64 * hsel;
        // causal: key j is visible to query i0 + e iff e >= j - L + Sq - i0
        const int qlo = p.causal ? j - it.L + p.Sq - i0 : -1;
        const float2* nlq = reinterpret_cast<const float2*>(nlv);
        const float4* ndg = reinterpret_cast<const float4*>(&c.ndel[s][64 * hsel]);
        const uint32_t ts = t_s + lane_off + 64 * hsel;
        float pr[64];
        tmem_ld64(ts, reinterpret_cast<uint32_t*>(pr));
        tc_fence_before();
        mbar_arrive_warp(&c.s_free);  // S^T(g)'s columns may take S^T(g + 1)
        // every query of this half visible to every key of the warp: no masking
        if (__all_sync(0xffffffffu, key_ok && qlo <= 0)) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float2 x = f2fma(make_float2(pr[2 * e], pr[2 * e + 1]), sl2, nlq[e]);
            pr[2 * e] = ex2_approx(x.x);
            pr[2 * e + 1] = ex2_approx(x.y);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float2 nl = nlq[e];
            const float x0 = fmaf(pr[2 * e], p.scale_log2, nl.x), x1 = fmaf(pr[2 * e + 1], p.scale_log2, nl.y);
            pr[2 * e] = key_ok && 2 * e >= qlo ? ex2_approx(x0) : 0.f;
            pr[2 * e + 1] = key_ok && 2 * e + 1 >= qlo ? ex2_approx(x1) : 0.f;
          }
        }
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) pk[e] = pack_bf16x2(pr[2 * e], pr[2 * e + 1]);
        // P^T(g) into the shared tile once dV(g - 1) has read P^T(g - 1) there: row r of
        // the 64-query chunk hsel, 16-byte unit u (queries 8 u .. 8 u + 7) at the
        // 128-byte-swizzled position u ^ (r mod 8)
        if (gt >= 1 && !wait_phase_warp(&c.dv_done, (gt - 1) & 1, wc)) { ok = false; break; }
        {
          uint8_t* prow = sP + hsel * kChunk + r * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(prow + ((u ^ (r & 7)) * 16)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
        fence_proxy_async_smem();
        mbar_arrive_warp(&c.p_ready);
        // dS^T = P^T * (dP^T - delta), over dP^T's first columns of this half; a key past
        // the valid length may turn NaN here, but its dK row is written as zeros. The
        // -delta of each 32-column half is fetched ahead of its use, as above.
        float4 ndv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) ndv[e] = ndg[e];
        if (!wait_phase_warp(&c.dp_full[gt % NDP], (gt / NDP) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tdp = t_dp + (gt % NDP) * 128 + lane_off + 64 * hsel;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float4 ndn[8];
          if (half == 0) {
#pragma unroll
            for (int e = 0; e < 8; ++e) ndn[e] = ndg[8 + e];
          }
          float dp[32];
          tmem_ld32(tdp + 32 * half, reinterpret_cast<uint32_t*>(dp));
          uint32_t dd[16];
          const float2* ndq = reinterpret_cast<const float2*>(ndv);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c0 = 32 * half + 2 * e;
            const float2 d = f2mul(f2add(make_float2(dp[2 * e], dp[2 * e + 1]), ndq[e]),
                                   make_float2(pr[c0], pr[c0 + 1]));
            dd[e] = pack_bf16x2(d.x, d.y);
          }
          tmem_st16(tdp + 16 * half, dd);
          if (half == 0) {
#pragma unroll
            for (int e = 0; e < 8; ++e) ndv[e] = ndn[e];
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(&c.ds_ready[gt % NDP]);
      }
      if (!ok) break;
      // epilogue: half 0 writes dV, half 1 writes dK (times the scale); rows past the
      // valid length are written as zeros
      if (!wait_phase_warp(&c.acc_done, item_cnt & 1, wc)) { ok = false; break; }
      tc_fence_after();
      __nv_bfloat16* dst = (hsel == 0 ? p.dv : p.dk) + orow;
      float* pdst = (hsel == 0 ? p.part_dv : p.part_dk) + prow;
      const uint32_t tacc = (hsel == 0 ? t_dv : t_dk) + lane_off;
      const float mul = hsel == 0 ? 1.f : p.scale;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        tmem_ld32(tacc + cc * 32, v);
        if (j < p.Skv) {
          if (p.split) {
            // this run of query heads' share, unscaled (the group reduction scales dK), in
            // 32-byte stores: the workspace rows are 256-byte aligned
            if (!key_ok) {
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = 0u;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) st_global_v8(pdst + cc * 32 + 8 * e, v + 8 * e);
          } else if (key_ok) {
            if (out32) store_row_bf16_v8(dst + cc * 32, v, mul);
            else store_row_bf16(dst + cc * 32, v, mul);
          } else {
            zero_row_bf16(dst + cc * 32, 32);
          }
        }
      }
      tc_fence_before();
      mbar_arrive_warp(&c.acc_free);
      ++item_cnt;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // this grid may start before the dQ grid it depends on programmatically has finished;
  // waiting for that grid before exiting makes the completion of this grid (which the
  // caller's later work on the stream waits for) imply the completion of the dQ grid. The
  // dQ grid is the shorter one, so the wait costs nothing in practice.
  griddep_wait();
}

// ========================================================================== delta
// delta[b, h, i] = sum_d dO[b, i, h, d] * O[b, i, h, d] (fp32), the row term of the
// softmax Jacobian; each row is read by D / 8 lanes, 16 bytes of O and dO each.
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        float* __restrict__ delta, int B, int Sq, int Hq) {
  constexpr int kG = D / 8;
  const int64_t rows = (int64_t)B * Sq * Hq;
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / kG;
  const int part = threadIdx.x % kG;
  float a = 0.f;
  if (row < rows) {
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(o + row * D) + part);
    const uint4 y = __ldg(reinterpret_cast<const uint4*>(dout + row * D) + part);
    a = fmaf(bf16_lo(x.x), bf16_lo(y.x), a); a = fmaf(bf16_hi(x.x), bf16_hi(y.x), a);
    a = fmaf(bf16_lo(x.y), bf16_lo(y.y), a); a = fmaf(bf16_hi(x.y), bf16_hi(y.y), a);
    a = fmaf(bf16_lo(x.z), bf16_lo(y.z), a); a = fmaf(bf16_hi(x.z), bf16_hi(y.z), a);
    a = fmaf(bf16_lo(x.w), bf16_lo(y.w), a); a = fmaf(bf16_hi(x.w), bf16_hi(y.w), a);
  }
#pragma unroll
  for (int m = 1; m < kG; m <<= 1) a += __shfl_xor_sync(0xffffffffu, a, m);
  if (part == 0 && row < rows) {
    const int h = (int)(row % Hq);
    const int64_t bi = row / Hq;  // b * Sq + i
    const int i = (int)(bi % Sq), b = (int)(bi / Sq);
    delta[((int64_t)b * Hq + h) * Sq + i] = a;
  }
}

// ===================================================================== group reduction
// Split mode: dK[b, j, kvh] = scale * sum over the group's parts r = 0 .. parts - 1 (in
// that order) of the partial dK[b, j, kvh * parts + r]; likewise dV (unscaled). Each
// thread reduces 4 consecutive elements of one (b, j, kvh) row.
__global__ void __launch_bounds__(256) bwd_group_reduce_kernel(const float* __restrict__ part_dk,
                                                               const float* __restrict__ part_dv,
                                                               __nv_bfloat16* dk, __nv_bfloat16* dv,
                                                               int B, int Skv, int Hkv, int parts, int D,
                                                               float scale) {
  // launched as a programmatic dependent of the dK/dV kernel: the partials are complete
  // and visible after this wait
  griddep_wait();
  const int64_t n4 = (int64_t)B * Skv * Hkv * D / 4;
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n4) return;
  const int d4 = (int)(e % (D / 4));
  const int64_t row = e / (D / 4);  // (b * Skv + j) * Hkv + kvh
  const int64_t src0 = row * parts * D + 4 * d4;
  float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sv = sk;
  for (int r = 0; r < parts; ++r) {
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
  return 2 * (size_t)kT * D * 2 + 2 * (size_t)NST * kT * D * 2 + (size_t)kT * kT * 2 + sizeof(DkvCtl<NST>);
}
template <int D, int NK, int NV>
constexpr size_t dq_smem() {
  return 1024 + (size_t)(2 + NK + NV) * kT * D * 2 + sizeof(DqCtl<NK, NV>);
}
// dK/dV: Q/dO stages of 128 queries, as many as fit in 227 KB next to K, V and P^T
template <int D>
constexpr int kStages = D == 64 ? 4 : 2;
static_assert(dkdv_smem<64, kStages<64>>() <= 232448 && dkdv_smem<128, kStages<128>>() <= 232448,
              "dK/dV shared memory");
// dQ: K and V rings
template <int D>
constexpr int kKStages = D == 64 ? 6 : 3;
template <int D>
constexpr int kVStages = D == 64 ? 5 : 2;
static_assert(dq_smem<64, kKStages<64>, kVStages<64>>() <= 232448 &&
                  dq_smem<128, kKStages<128>, kVStages<128>>() <= 232448,
              "dQ shared memory");

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
  constexpr int NST = kStages<D>;
  BwdParams prm{};
  const bool no_keys = p.Skv == 0;
  // every tile is 128 rows: Q and dO of 128 queries, K and V of 128 keys
  if (!make_bshd_map(&prm.tm_q, p.q, p.B, p.Sq, p.Hq, D, kT) ||
      !make_bshd_map(&prm.tm_do, p.dout, p.B, p.Sq, p.Hq, D, kT) ||
      !make_bshd_map(&prm.tm_k, no_keys ? p.q : p.k, p.B, no_keys ? p.Sq : p.Skv,
                     no_keys ? p.Hq : p.Hkv, D, kT) ||
      !make_bshd_map(&prm.tm_v, no_keys ? p.q : p.v, p.B, no_keys ? p.Sq : p.Skv,
                     no_keys ? p.Hq : p.Hkv, D, kT))
    return cudaErrorInvalidValue;
  prm.o = static_cast<const __nv_bfloat16*>(p.o_in);
  prm.dout = static_cast<const __nv_bfloat16*>(p.dout);
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
  {
    const int g = p.Hq / p.Hkv, gs = p.split ? p.split : 1;
    const int n_qt = (p.Sq + kT - 1) / kT, n_kt = (p.Skv + kT - 1) / kT;
    prm.fd_bh = FastDiv::make(p.B * p.Hq);
    prm.fd_hq = FastDiv::make(p.Hq);
    prm.fd_nqt = FastDiv::make(n_qt);
    prm.fd_g = FastDiv::make(g);
    prm.fd_bkgs = FastDiv::make(p.B * p.Hkv * gs);
    prm.fd_ktgs = FastDiv::make(n_kt * gs);
    prm.fd_gs = FastDiv::make(gs);
    prm.fd_hkv = FastDiv::make(p.Hkv);
    prm.heads_per_item = g / gs;
  }
  const int sms = g_num_sms[dev];
  {
    const int64_t threads = (int64_t)p.B * p.Sq * p.Hq * (D / 8);
    if (threads > 0) {
      bwd_delta_kernel<D><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(
          prm.o, prm.dout, prm.delta, p.B, p.Sq, p.Hq);
      count_launches(1);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  prm.n_items = p.B * p.Hq * ((p.Sq + kT - 1) / kT);
  {
    constexpr int NK = kKStages<D>, NV = kVStages<D>;
    constexpr size_t smem = dq_smem<D, NK, NV>();
    cudaError_t e = set_smem(bwd_dq_sm103_kernel<D, NK, NV>, smem, dev, D == 64 ? 2 : 3);
    if (e != cudaSuccess) return e;
    bwd_dq_sm103_kernel<D, NK, NV><<<prm.n_items < sms ? prm.n_items : sms, kThreads, smem, s>>>(prm);
    count_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (p.Skv > 0) {
    prm.n_items = p.B * p.Hkv * ((p.Skv + kT - 1) / kT) * (p.split ? p.split : 1);
    constexpr size_t smem = dkdv_smem<D, NST>();
    cudaError_t e = set_smem(bwd_dkdv_sm103_kernel<D, NST>, smem, dev, D == 64 ? 0 : 1);
    if (e != cudaSuccess) return e;
    // a programmatic dependent of the dQ kernel: both only read Q, K, V, dO, LSE and delta
    // (complete before the dQ kernel started) and write disjoint outputs, so the dK/dV
    // CTAs need not wait for the dQ grid to finish
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(prm.n_items < sms ? prm.n_items : sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, bwd_dkdv_sm103_kernel<D, NST>, prm);
    if (e != cudaSuccess) return e;
    count_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.split) {
      const int64_t n4 = (int64_t)p.B * p.Skv * p.Hkv * D / 4;
      cudaLaunchAttribute rattr[1];
      rattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      rattr[0].val.programmaticStreamSerializationAllowed = 1;
      cudaLaunchConfig_t rcfg{};
      rcfg.gridDim = dim3((unsigned)((n4 + 255) / 256));
      rcfg.blockDim = dim3(256);
      rcfg.stream = s;
      rcfg.attrs = rattr;
      rcfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&rcfg, bwd_group_reduce_kernel, static_cast<const float*>(p.part_dk),
                             static_cast<const float*>(p.part_dv), prm.dk, prm.dv, p.B, p.Skv, p.Hkv,
                             p.split, D, p.scale);
      if (e != cudaSuccess) return e;
      count_launches(1);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
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
  return p.D == 64 ? launch_bwd<64>(p, dev, s) : launch_bwd<128>(p, dev, s);
}

}  // namespace attn
