// bf16 attention forward for sm_103a: TMA -> shared memory, tcgen05.mma -> TMEM,
// online softmax in registers, P back to TMEM as the A operand of the PV product.
//
// The computation is the fused flash forward of "xtrain evolution.md" (infrastructure
// table, row T14: online softmax tiled over K/V, the N x N scores never materialised),
// with GQA heads sharing K/V (row T15) and varlen keys: keys at or past the valid length
// are padding and never enter a result ("LingBot full-pipeline analysis report", section
// "same-GPU FA2/FA3 hardware comparison").
//
// One persistent CTA per SM (384 threads) loops over work items of 256 query rows of one
// (batch, head), taken in a longest-first order:
//   warp 0      TMA producer: a ring of Q tiles (the next item's Q is prefetched), and a
//               ring of K/V tiles of 128 keys;
//   warps 1, 2  MMA issuers (one thread each, one per Q tile): S_t = Q_t K^T into TMEM,
//               O_t += P_t V from TMEM;
//   warp 3      zeroes the padding rows of partial V tiles;
//   warps 4-7   softmax of Q tile 0 (128 rows, one row per thread);
//   warps 8-11  softmax of Q tile 1.
// TMEM (512 columns): S0 | S1 | O0 | O1. The softmax reads its S row, writes P (bf16)
// over the first half of the same columns, and the PV MMA reads P from there. A row's
// running max is only raised (and O, l rescaled) when it grows by more than 2^8, which
// leaves the result exact while skipping almost every rescale.
//
// Every barrier wait is bounded in time; a wait that runs out flags ATTN_DEVERR_TIMEOUT,
// makes the whole CTA give up, waits (bounded) for its own copies and MMAs in flight,
// frees its TMEM and returns.

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

constexpr int kBM = 128;         // rows of a Q tile (TMEM lanes)
constexpr int kBN = 128;         // keys of a K/V tile
constexpr int kItemRows = 2 * kBM;
constexpr int kThreads = 384;    // warps 0-3: producer, 2 MMA issuers, V fixer; 4-7, 8-11: softmax
// Register split (setmaxnreg): the block launches with kLaunchRegs a thread; warpgroup 0
// then drops to kRegsLow and the two softmax warpgroups rise to kRegsHigh. The raise
// draws on the registers the block was launched with, so the split must fit in them.
constexpr int kLaunchRegs = 168;
constexpr int kRegsLow = 112;
constexpr int kRegsHigh = 192;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * kLaunchRegs, "register split");
constexpr int kMaxSortedHeads = 64;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows > 2^8

struct FwdParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  __nv_bfloat16* o;
  float* lse;
  const int32_t* kv_lens;
  unsigned int* err;
  int B, Hq, Hkv, Sq, Skv;
  int causal;
  int head_inner;    // non-causal order with the (batch, head) index innermost
  int n_qblocks;
  int n_items;
  float scale_log2;  // scale * log2(e)
  uint64_t timeout_ns;
  uint32_t fault;    // test-only: bit 0 = the producer of CTA 0 skips its first K load
};

template <int NQ, int NST>
struct FwdCtl {
  uint64_t mma_final[2];
  uint64_t q_full[NQ], q_empty[NQ];
  uint64_t kv_full[NST], kv_empty[NST], kv_fixed[NST], fix_req[NST];
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
  uint32_t tmem_base;
  int abort;
  int n_sorted;
  int sorted[kMaxSortedHeads];
  int lens[kMaxSortedHeads];
};

struct Item {
  int b, h, kvh, q0, L;
  int n[2];   // K/V tiles each Q tile visits
  int nload;  // K/V tiles loaded (max of n)
};

__device__ __forceinline__ int clamp_len(int L, int Skv) { return L < 0 ? 0 : (L > Skv ? Skv : L); }

template <typename Ctl>
__device__ __forceinline__ Item decode_item(int idx, const FwdParams& p, const Ctl& c) {
  const int g = p.Hq / p.Hkv;
  int b, h, qb;
  if (p.causal) {
    // longest first: the last query blocks see the most keys
    const int BH = p.B * p.Hq;
    qb = p.n_qblocks - 1 - idx / BH;
    const int bh = idx % BH;
    b = bh / p.Hq;
    h = bh % p.Hq;
  } else if (c.n_sorted > 0) {
    // varlen: (batch, kv head) groups in decreasing valid length
    const int per = g * p.n_qblocks;
    const int bk = c.sorted[idx / per];
    const int rem = idx % per;
    b = bk / p.Hkv;
    h = (bk % p.Hkv) * g + rem / p.n_qblocks;
    qb = rem % p.n_qblocks;
  } else if (p.head_inner) {
    // short K/V (L2-resident): concurrent CTAs cover every head of the same query rows,
    // so Q is read and O written as whole contiguous rows across heads
    const int BH = p.B * p.Hq;
    qb = idx / BH;
    const int bh = idx % BH;
    b = bh / p.Hq;
    h = bh % p.Hq;
  } else {
    // long K/V: consecutive query blocks of one head run together and share K/V in L2
    const int bh = idx / p.n_qblocks;
    qb = idx % p.n_qblocks;
    b = bh / p.Hq;
    h = bh % p.Hq;
  }
  Item it;
  it.b = b;
  it.h = h;
  it.kvh = h / g;
  it.q0 = qb * kItemRows;
  it.L = p.kv_lens ? clamp_len(__ldg(p.kv_lens + b * p.Hkv + it.kvh), p.Skv) : p.Skv;
  it.nload = 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int i0 = it.q0 + t * kBM;
    int n = 0;
    if (i0 < p.Sq) {
      int kmax = it.L;
      if (p.causal) {
        const int ilast = min(i0 + kBM - 1, p.Sq - 1);
        kmax = min(it.L, ilast + it.L - p.Sq + 1);
      }
      kmax = max(kmax, 0);
      n = (kmax + kBN - 1) / kBN;
    }
    it.n[t] = n;
    it.nload = max(it.nload, n);
  }
  return it;
}

// Whether K/V tile j holds in-bounds rows at or past the valid length (padding that may
// hold anything, even NaN): such a V tile gets those rows zeroed before the PV product.
__device__ __forceinline__ bool needs_fix(int j, int L, int Skv) {
  return min(Skv, (j + 1) * kBN) > L;
}

// Number of 16-key steps of the PV product for tile j: only steps holding valid keys.
__device__ __forceinline__ int pv_steps(int j, int L) {
  const int valid = min(kBN, L - j * kBN);
  return (valid + 15) / 16;
}

template <int D, int NQ, int NST>
// 12 warps, 3 per sub-partition (16K registers each): launched with <= 168 registers a
// thread, then rebalanced with setmaxnreg (see kRegsLow / kRegsHigh).
__global__ void __launch_bounds__(kThreads, 1) fwd_sm103_kernel(const __grid_constant__ FwdParams p) {
  constexpr int kQTile = kBM * D * 2;     // bytes of a Q tile
  constexpr int kKVTile = kBN * D * 2;    // bytes of a K or V tile
  constexpr int kQChunk = kBM * 128;      // 64 columns (128 bytes) of a Q tile
  constexpr int kKVChunk = kBN * 128;
  constexpr int kChunks = D / 64;
  constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, false, true);
  using Ctl = FwdCtl<NQ, NST>;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                    // NQ tile slots
  uint8_t* sKV = smem + NQ * kQTile;     // NST tile slots
  Ctl& c = *reinterpret_cast<Ctl*>(sKV + NST * kKVTile);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // ------------------------------------------------------------------- prologue
  if (threadIdx.x == 0) {
    mbar_init(&c.mma_final[0], 1);
    mbar_init(&c.mma_final[1], 1);
    for (int s = 0; s < NQ; ++s) {
      mbar_init(&c.q_full[s], 1);
      mbar_init(&c.q_empty[s], 1);
    }
    for (int s = 0; s < NST; ++s) {
      mbar_init(&c.kv_full[s], 1);
      mbar_init(&c.kv_empty[s], 2);  // released by both MMA issuers
      mbar_init(&c.kv_fixed[s], 1);
      mbar_init(&c.fix_req[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&c.s_full[t], 1);
      mbar_init(&c.p_full[t], kBM);
      mbar_init(&c.o_done[t], 1);
      mbar_init(&c.o_free[t], kBM);
    }
    c.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&c.tmem_base, 512);
    tmem_relinquish();
  }
  // varlen order: rank the (batch, kv head) groups by decreasing valid length
  const int nbk = p.B * p.Hkv;
  const bool sort_heads = !p.causal && p.kv_lens != nullptr && nbk <= kMaxSortedHeads;
  if (p.kv_lens != nullptr) {
    for (int e = threadIdx.x; e < nbk; e += kThreads) {
      const int raw = __ldg(p.kv_lens + e);
      if ((raw < 0 || raw > p.Skv) && blockIdx.x == 0) atomicOr(p.err, ATTN_DEVERR_KVLEN);
      if (sort_heads) c.lens[e] = clamp_len(raw, p.Skv);
    }
  }
  __syncthreads();
  if (sort_heads) {
    for (int e = threadIdx.x; e < nbk; e += kThreads) {
      const int Le = c.lens[e];
      int rank = 0;
      for (int f = 0; f < nbk; ++f) {
        const int Lf = c.lens[f];
        rank += (Lf > Le) || (Lf == Le && f < e);
      }
      c.sorted[rank] = e;
    }
  }
  if (threadIdx.x == 0) c.n_sorted = sort_heads ? nbk : 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  WaitCtl wc{&c.abort, p.err, p.timeout_ns};

  if (warp < 4) {
    // warpgroup 0 hands registers to the softmax warpgroups
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegsLow) : "memory");
    if (warp == 0) {
      // ------------------------------------------------------------- TMA producer
      if (lane == 0) {
        tma_prefetch_map(&p.tm_q);
        tma_prefetch_map(&p.tm_k);
        tma_prefetch_map(&p.tm_v);
      }
      uint32_t slot = 0, ring_par = 0, qs = 0, q_par = 0;
      uint32_t issued = 0, last_par = 0;    // per K/V slot: a load was issued / its parity
      uint32_t q_issued = 0, q_last = 0;    // per Q slot
      bool ok = true, first = true;
      for (int idx = blockIdx.x; ok && idx < p.n_items; idx += gridDim.x) {
        const Item it = decode_item(idx, p, c);
        if (it.nload == 0) continue;
        for (int t = 0; t < 2; ++t) {
          if (!wait_phase_warp(&c.q_empty[qs], q_par ^ 1, wc)) { ok = false; break; }
          if (lane == 0) {
            mbar_expect_tx(&c.q_full[qs], kQTile);
            for (int ch = 0; ch < kChunks; ++ch)
              tma_load_4d(sQ + qs * kQTile + ch * kQChunk, &p.tm_q, &c.q_full[qs], ch * 64, it.h,
                          it.q0 + t * kBM, it.b);
          }
          q_issued |= 1u << qs;
          q_last = (q_last & ~(1u << qs)) | (q_par << qs);
          if (++qs == NQ) { qs = 0; q_par ^= 1; }
        }
        for (int j = 0; ok && j < it.nload; ++j) {
          for (int kv = 0; kv < 2; ++kv) {
            if (!wait_phase_warp(&c.kv_empty[slot], ring_par ^ 1, wc)) { ok = false; break; }
            const bool skip = (p.fault & 1u) && blockIdx.x == 0 && first && j == 0 && kv == 0;
            if (!skip) {
              if (lane == 0) {
                mbar_expect_tx(&c.kv_full[slot], kKVTile);
                for (int ch = 0; ch < kChunks; ++ch)
                  tma_load_4d(sKV + slot * kKVTile + ch * kKVChunk, kv == 0 ? &p.tm_k : &p.tm_v,
                              &c.kv_full[slot], ch * 64, it.kvh, j * kBN, it.b);
              }
              issued |= 1u << slot;
              last_par = (last_par & ~(1u << slot)) | (ring_par << slot);
            }
            // a V tile with padding rows: warp 3 zeroes them once the tile has landed
            if (kv == 1 && needs_fix(j, it.L, p.Skv) && lane == 0) mbar_arrive(&c.fix_req[slot]);
            if (++slot == NST) { slot = 0; ring_par ^= 1; }
          }
        }
        first = false;
      }
      // every copy this CTA started lands before its shared memory can go away (after an
      // abort the consumers may never have waited for them)
      for (int s = 0; s < NST; ++s)
        if (issued & (1u << s)) wait_phase_teardown(&c.kv_full[s], (last_par >> s) & 1, 200000000ull);
      for (int s = 0; s < NQ; ++s)
        if (q_issued & (1u << s)) wait_phase_teardown(&c.q_full[s], (q_last >> s) & 1, 200000000ull);
    } else if (warp == 1 || warp == 2) {
      // ------------------------------------------------------------- MMA issuers
      // one issuing thread per Q tile (warp 1: tile 0, warp 2: tile 1), so that each
      // tile's S / PV chain advances as soon as its own softmax is done; both threads
      // release every K/V slot (kv_empty counts two arrivals)
      if (lane == 0) {
        const int t = warp - 1;
        const uint32_t sQa = smem_u32(sQ), sKVa = smem_u32(sKV);
        // K-major Q and K tiles (128-byte rows, 8-row groups 1024 bytes apart); MN-major V
        // (64-column chunks kKVChunk bytes apart)
        const uint64_t desc_q0 = smem_desc_sw128(sQa, 16, 1024);
        const uint64_t desc_k0 = smem_desc_sw128(sKVa, 16, 1024);
        const uint64_t desc_v0 = smem_desc_sw128(sKVa, kKVChunk, 1024);
        // ring positions: the k-th loaded item's Q tile t is Q position 2 k + t; its K/V
        // tile j is at 2 (kbase + j) (K) and 2 (kbase + j) + 1 (V); a position's slot is
        // pos % N and its phase parity (pos / N) % 2
        uint32_t kbase = 0, qpos = t, fix_par = 0, pv = 0, pc = 0, ic = 0;
        bool ok = true;
        for (int idx = blockIdx.x; ok && idx < p.n_items; idx += gridDim.x) {
          const Item it = decode_item(idx, p, c);
          if (it.nload == 0) continue;
          const int nt = t == 0 ? it.n[0] : it.n[1];
          const uint32_t qslot = qpos % NQ;
          if (!wait_phase(&c.q_full[qslot], (qpos / NQ) & 1, wc)) { ok = false; break; }
          qpos += 2;
          tc_fence_after();
          if (nt == 0) mma_commit(&c.q_empty[qslot]);  // never read: free at once
          for (int j = 0; ok && j < it.nload; ++j) {
            const uint32_t kpos = 2 * (kbase + j), vpos = kpos + 1;
            const uint32_t ks = kpos % NST, vs = vpos % NST;
            // S_t(j) = Q_t K_j^T; S_t's columns hold P_t(j - 1) until PV_t(j - 1) completes
            if (!wait_phase(&c.kv_full[ks], (kpos / NST) & 1, wc)) { ok = false; break; }
            if (j < nt) {
              if (pv > 0 && !wait_phase(&c.o_done[t], (pv - 1) & 1, wc)) { ok = false; break; }
              tc_fence_after();
              const uint64_t a0 = desc_q0 + ((qslot * kQTile) >> 4);
              const uint64_t b0 = desc_k0 + ((ks * kKVTile) >> 4);
  #pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                mma_ss(tmem + t * 128, a0 + (((kk / 4) * kQChunk + (kk % 4) * 32) >> 4),
                       b0 + (((kk / 4) * kKVChunk + (kk % 4) * 32) >> 4), kIdescS, kk > 0 ? 1u : 0u);
              }
              mma_commit(&c.s_full[t]);
              if (j == nt - 1) mma_commit(&c.q_empty[qslot]);  // last read of Q_t
            }
            mma_commit(&c.kv_empty[ks]);
            // O_t += P_t(j) V_j
            if (needs_fix(j, it.L, p.Skv)) {
              if (!wait_phase(&c.kv_fixed[vs], (fix_par >> vs) & 1, wc)) { ok = false; break; }
              fix_par ^= 1u << vs;
            } else if (!wait_phase(&c.kv_full[vs], (vpos / NST) & 1, wc)) {
              ok = false;
              break;
            }
            if (j < nt) {
              if (!wait_phase(&c.p_full[t], pc & 1, wc)) { ok = false; break; }
              ++pc;
              if (j == 0 && !wait_phase(&c.o_free[t], (ic & 1) ^ 1, wc)) { ok = false; break; }
              tc_fence_after();
              const int steps = pv_steps(j, it.L);
              const uint64_t b0 = desc_v0 + ((vs * kKVTile) >> 4);
  #pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk) {
                if (kk < steps)
                  mma_ts(tmem + 256 + t * D, tmem + t * 128 + kk * 8, b0 + ((kk * 16 * 128) >> 4),
                         kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
              }
              mma_commit(&c.o_done[t]);
              ++pv;
            }
            mma_commit(&c.kv_empty[vs]);
          }
          if (!ok) break;
          kbase += it.nload;
          if (nt > 0) ++ic;
        }
        // every MMA this thread issued must finish before the TMEM is freed
        mma_commit(&c.mma_final[t]);
        wait_phase_teardown(&c.mma_final[t], 0, 200000000ull);
      }
      __syncwarp();
    } else {
      // -------------------------------------------------------------- V-tile fixer
      // zeroes the padding rows (at or past the valid length) of partial V tiles, so
      // that 0 * NaN in the PV product cannot occur; requests come from the producer
      // in ring order (fix_req), so the fill this waits for is never ambiguous
      uint32_t kbase = 0, fr_par = 0;
      bool ok = true;
      for (int idx = blockIdx.x; ok && idx < p.n_items; idx += gridDim.x) {
        const Item it = decode_item(idx, p, c);
        if (it.nload == 0) continue;
        for (int j = 0; j < it.nload; ++j) {
          if (!needs_fix(j, it.L, p.Skv)) continue;
          const uint32_t vpos = 2 * (kbase + j) + 1, vs = vpos % NST;
          if (!wait_phase_warp(&c.fix_req[vs], (fr_par >> vs) & 1, wc)) { ok = false; break; }
          fr_par ^= 1u << vs;
          if (!wait_phase_warp(&c.kv_full[vs], (vpos / NST) & 1, wc)) { ok = false; break; }
          const int r0 = it.L - j * kBN;  // first padding row (>= 1: tile j holds valid keys)
          const int units = (kBN - r0) * kChunks * 8;
          uint8_t* base = sKV + vs * kKVTile;
          for (int e = lane; e < units; e += 32) {
            const int r = r0 + e / (kChunks * 8);
            const int rest = e % (kChunks * 8);
            *reinterpret_cast<uint4*>(base + (rest / 8) * kKVChunk + r * 128 + (rest % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&c.kv_fixed[vs]);
        }
        kbase += it.nload;
      }
  }
  } else {
    // --------------------------------------------------------------------- softmax
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegsHigh) : "memory");
    const int t = (warp - 4) / 4;
    const int quad = warp % 4;  // TMEM lanes a warp may touch: 32 * (warp % 4) ...
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tO = tmem + lane_off + 256 + t * D;
    const bool pos_scale = p.scale_log2 > 0.f;
    uint32_t s_cnt = 0, npv = 0;
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < p.n_items; idx += gridDim.x) {
      const Item it = decode_item(idx, p, c);
      const int i = it.q0 + t * kBM + r;
      const bool row_ok = i < p.Sq;
      __nv_bfloat16* orow = p.o + ((static_cast<int64_t>(it.b) * p.Sq + i) * p.Hq + it.h) * D;
      float* lrow = p.lse + (static_cast<int64_t>(it.b) * p.Hq + it.h) * p.Sq + i;
      const int nt = t == 0 ? it.n[0] : it.n[1];
      if (nt == 0) {
        if (row_ok) {
          for (int d = 0; d < D; d += 8)
            *reinterpret_cast<uint4*>(orow + d) = make_uint4(0u, 0u, 0u, 0u);
          *lrow = -CUDART_INF_F;
        }
        continue;
      }
      // visible keys of this row: [0, kend)
      const int kend = p.causal ? min(it.L, i + it.L - p.Sq + 1) : it.L;
      float m = -CUDART_INF_F, l = 0.f;
      for (int j = 0; j < nt; ++j) {
        if (!wait_phase_warp(&c.s_full[t], s_cnt & 1, wc)) { ok = false; break; }
        ++s_cnt;
        tc_fence_after();
        const int limit = kend - j * kBN;
        // one TMEM round trip: the whole S row of this tile into registers
        float s[kBN];
        tmem_ld128(tS, reinterpret_cast<uint32_t*>(s));
        // the row max of the scaled scores over the visible keys, 8 independent chains;
        // for a positive scale the max of the raw scores, scaled once
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = -CUDART_INF_F;
        const bool full = limit >= kBN;
        if (pos_scale && full) {
#pragma unroll
          for (int e = 0; e < kBN / 2; ++e) mx8[e % 8] = max3f(mx8[e % 8], s[2 * e], s[2 * e + 1]);
        } else {
#pragma unroll
          for (int e = 0; e < kBN; ++e) {
            const float v = pos_scale ? s[e] : s[e] * p.scale_log2;
            mx8[e % 8] = fmaxf(mx8[e % 8], e < limit ? v : -CUDART_INF_F);
          }
        }
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const float mnew = fmaxf(m, pos_scale ? mx * p.scale_log2 : mx);
        const bool raise = mnew > m + kRescaleThreshold;
        const bool rescale = raise && m != -CUDART_INF_F;
        // TMEM loads/stores are warp-collective: the warp rescales together, rows that
        // need no rescale with a factor of 1. S_t(j) landed, so every earlier MMA of the
        // issuer (PV_t(j-1)) has too and O_t holds its sum.
        if (__any_sync(0xffffffffu, rescale)) {
          const float alpha = rescale ? ex2_approx(m - mnew) : 1.f;
          l *= alpha;
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t ov[32];
            tmem_ld32(tO + cc * 32, ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(tO + cc * 32, ov);
          }
        }
        if (raise) m = mnew;
        // P = 2^(s * scale * log2 e - m) in bf16 over the first half of S's columns, a
        // quarter at a time (the fence keeps each quarter after the previous store)
        const float msub = m == -CUDART_INF_F ? 0.f : m;
        float rs8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) rs8[e] = 0.f;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t pk[16];
          if (q4 > 0) reg_fence32(s + q4 * 32);  // after the previous quarter's store
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c0 = q4 * 32 + 2 * e;
            float x0, x1;
            ffma2_bcast(x0, x1, s[c0], s[c0 + 1], p.scale_log2, -msub);
            if (!full) {
              x0 = c0 < limit ? x0 : -CUDART_INF_F;
              x1 = c0 + 1 < limit ? x1 : -CUDART_INF_F;
            }
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            fadd2_acc(rs8[2 * (e % 4)], rs8[2 * (e % 4) + 1], p0, p1);
            pk[e] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tS + q4 * 16, pk);
        }
        l += ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&c.p_full[t]);
        ++npv;
      }
      if (!ok) break;
      // epilogue: O / l and LSE
      if (!wait_phase_warp(&c.o_done[t], (npv - 1) & 1, wc)) { ok = false; break; }
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t ov[32];
        tmem_ld32(tO + cc * 32, ov);
        if (row_ok) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
      if (row_ok) *lrow = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
      tc_fence_before();
      mbar_arrive(&c.o_free[t]);
    }
  }

  // ---------------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------- host side
template <int D, int NQ, int NST>
constexpr size_t fwd_smem_bytes() {
  return 1024 + (size_t)NQ * kBM * D * 2 + (size_t)NST * kBN * D * 2 + sizeof(FwdCtl<NQ, NST>);
}

constexpr int kMaxDev = 64;
std::mutex g_mu;
int g_num_sms[kMaxDev] = {};
bool g_attr_set[kMaxDev][2] = {};

template <int D, int NQ, int NST>
cudaError_t launch(const FwdParams& prm, int dev, cudaStream_t s) {
  constexpr size_t smem = fwd_smem_bytes<D, NQ, NST>();
  static_assert(smem <= 232448, "shared memory per block");
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const int which = D == 64 ? 0 : 1;
    if (!g_attr_set[dev][which]) {
      // the register split is only safe if the block launches with enough registers:
      // a raise that the launch allocation cannot cover would wait forever
      cudaFuncAttributes fa;
      cudaError_t e = cudaFuncGetAttributes(&fa, fwd_sm103_kernel<D, NQ, NST>);
      if (e != cudaSuccess) return e;
      if (fa.numRegs * kThreads < 128 * kRegsLow + 256 * kRegsHigh || fa.numRegs > kLaunchRegs)
        return cudaErrorInvalidConfiguration;
      e = cudaFuncSetAttribute(fwd_sm103_kernel<D, NQ, NST>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      g_attr_set[dev][which] = true;
    }
  }
  const int grid = prm.n_items < g_num_sms[dev] ? prm.n_items : g_num_sms[dev];
  fwd_sm103_kernel<D, NQ, NST><<<grid, kThreads, smem, s>>>(prm);
  count_launches(1);
  return cudaGetLastError();
}

uint32_t g_fault_next = 0;
uint64_t g_fault_timeout_ns = 0;

}  // namespace

namespace {
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
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}
}  // namespace

bool make_bshd_map(CUtensorMap* map, const void* base, int B, int S, int H, int D, int rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2,
                                 (cuuint64_t)S * H * D * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void tc_set_test_fault(uint32_t mask, uint64_t timeout_ns) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_fault_next = mask;
  g_fault_timeout_ns = timeout_ns;
}

cudaError_t tc_fwd(const Problem& p, cudaStream_t s) {
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
  FwdParams prm{};
  // with no keys the K/V maps are never used; describe q so that encoding succeeds
  const bool no_keys = p.Skv == 0;
  if (!make_bshd_map(&prm.tm_q, p.q, p.B, p.Sq, p.Hq, p.D, kBM) ||
      !make_bshd_map(&prm.tm_k, no_keys ? p.q : p.k, p.B, no_keys ? p.Sq : p.Skv,
                no_keys ? p.Hq : p.Hkv, p.D, kBN) ||
      !make_bshd_map(&prm.tm_v, no_keys ? p.q : p.v, p.B, no_keys ? p.Sq : p.Skv,
                no_keys ? p.Hq : p.Hkv, p.D, kBN))
    return cudaErrorInvalidValue;
  prm.o = static_cast<__nv_bfloat16*>(p.o);
  prm.lse = p.lse;
  prm.kv_lens = p.kv_lens;
  prm.err = p.err;
  prm.B = p.B;
  prm.Hq = p.Hq;
  prm.Hkv = p.Hkv;
  prm.Sq = p.Sq;
  prm.Skv = p.Skv;
  prm.causal = p.causal;
  // K/V of every head small enough to stay in L2 (a third of its 129 MB)
  prm.head_inner = (double)p.B * p.Hkv * p.Skv * p.D * 2 * 2 <= 43.0e6 ? 1 : 0;
  prm.n_qblocks = (p.Sq + kItemRows - 1) / kItemRows;
  prm.n_items = p.B * p.Hq * prm.n_qblocks;
  prm.scale_log2 = p.scale * 1.4426950408889634f;
  prm.timeout_ns = 4000000000ull;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    prm.fault = g_fault_next;
    if (g_fault_next != 0 && g_fault_timeout_ns != 0) prm.timeout_ns = g_fault_timeout_ns;
    g_fault_next = 0;
  }
  if (p.D == 64) return launch<64, 4, 8>(prm, dev, s);
  return launch<128, 3, 4>(prm, dev, s);
}

}  // namespace attn
