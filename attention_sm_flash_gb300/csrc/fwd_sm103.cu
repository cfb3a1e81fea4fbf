// bf16 attention forward for sm_103a: TMA -> shared memory, tcgen05.mma -> TMEM,
// online softmax in registers, P back to TMEM as the A operand of the PV product.
//
// The computation is the fused flash forward of "xtrain evolution.md" (infrastructure
// table, row T14: online softmax tiled over K/V, the N x N scores never materialised),
// with GQA heads sharing K/V (row T15) and varlen keys: keys at or past the valid length
// are padding and never enter a result ("LingBot full-pipeline analysis report", section
// "same-GPU FA2/FA3 hardware comparison").
//
// One persistent CTA per SM (384 threads) loops over work items of 128 query rows (one Q
// tile) of one (batch, head), listed longest first and dealt to the CTAs in a snake order
// (round robin in the paged kind):
//   warp 0      TMA producer: a ring of Q tiles (the next item's Q is prefetched), and a
//               ring of K/V tiles of 128 keys;
//   warp 1      issues S = Q K^T into TMEM (one thread);
//   warp 2      zeroes the padding rows of partial V tiles;
//   warp 3      issues O += P V with P from TMEM (one thread);
//   warps 4-11  softmax, two threads per row (64 key columns each).
// TMEM (512 columns): S double buffer | P | O. S(j + 2) is computed into S(j)'s buffer as
// soon as the softmax has read S(j) into registers, so the softmax of tile j + 1 starts
// the moment tile j is done and the S products run under the softmax; P has its own
// columns, so no S product waits for a PV product, and the softmax only waits for
// PV(j - 1) before it overwrites P. (Two Q tiles per CTA with P written over S, the
// layout that fits two tiles in TMEM, measured 40 % tensor-pipe use: each S waited for
// the previous PV of its tile, and the two tiles' chains ran in lockstep.) A row's
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
#include "fastdiv.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

using namespace sm103;

constexpr int kBM = 128;         // rows of a Q tile (TMEM lanes)
constexpr int kBN = 128;         // keys of a K/V tile
constexpr int kItemRows = kBM;
constexpr int kThreads = 384;    // warps 0-3: producer, S issuer, V fixer, PV issuer; 4-11: softmax
constexpr int kSoftThreads = 256;
// registers a thread at launch (the most a 384-thread block gets), and the split of them
// between the control warpgroup and the two softmax warpgroups
constexpr int kRegsLaunch = 168, kRegsCtl = 152, kRegsSoft = 176;
constexpr int kMaxSortedHeads = 64;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows > 2^8
// Kernel kinds, a template parameter so that each is compiled without the others' code:
// dense K/V, a paged K/V cache, and split-KV items writing partials.
constexpr int kDense = 0, kPaged = 1, kSplit = 2;

struct FwdParams {
  CUtensorMap tm_q;
  CUtensorMap tm_o;  // O, same layout and box as Q (the epilogue's tile stores)
  CUtensorMap tm_k;  // dense [B, Skv, Hkv, D], or the page pool [pages, page_size, Hkv, D]
  CUtensorMap tm_v;
  __nv_bfloat16* o;
  float* lse;
  const int32_t* kv_lens;
  int lens_bstride, lens_hstride;  // valid length of (b, kvh) = kv_lens[b * bs + kvh * hs]
  unsigned int* err;
  // paged K/V (block_table non-null): key t of sequence b is row t % page_size of page
  // block_table[b * max_pages + t / page_size]; Skv = max_pages * page_size
  const int32_t* block_table;
  int max_pages, num_pages;
  // page_size = 1 << page_shift; page_box = 1 << box_shift rows per TMA box. Powers of two,
  // so the producer works with shifts: an integer division by a runtime value needs the
  // MUFU reciprocal, whose queue the softmax's exponentials keep full (measured: several
  // hundred cycles per box on the producer's critical path)
  int page_shift, box_shift;
  // split-KV: each (b, h, q block) is n_splits items over consecutive ranges of
  // split_tiles key tiles; an item writes its normalised partial O and LSE (fp32) and
  // fwd_combine_kernel merges them
  int n_splits, split_tiles;
  float* o_part;    // [n_splits, B, Hq, Sq, D]
  float* lse_part;  // [n_splits, B, Hq, Sq]
  int B, Hq, Hkv, Sq, Skv;
  // the divisions of the work decode, as multiplies (fastdiv.h): by the items of one
  // key range (n_items / n_splits), B * Hq, Hq, Hkv, n_qblocks, the GQA group
  // g = Hq / Hkv and g * n_qblocks
  FastDiv fd_range, fd_bh, fd_hq, fd_hkv, fd_qb, fd_g, fd_per;
  int causal;
  int head_inner;    // non-causal order with the (batch, head) index innermost
  int n_qblocks;
  int n_items;
  float scale_log2;  // scale * log2(e)
  uint64_t timeout_ns;
  uint32_t fault;    // test-only: bit 0 = the producer of CTA 0 skips its first K load
};

template <int NQ, int NK, int NV>
struct FwdCtl {
  uint64_t mma_final[2];
  uint64_t q_full[NQ], q_empty[NQ];
  uint64_t k_full[NK], k_empty[NK];
  uint64_t v_full[NV], v_empty[NV], v_fixed[NV], fix_req[NV];
  // per S/P buffer; a parity wait only tells apart phases one apart, and the softmax
  // can run two tiles ahead of the issuer, so P readiness is tracked per P buffer
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2], o_free;
  uint64_t xfull[4], xdone[4];  // per lane quadrant: the two threads of a row trade a value
  uint64_t o_staged, stage_free;  // the O staging tile: written by the softmax / read by TMA
  uint32_t tmem_base;
  int abort;
  float xbuf[2][kBM];           // [half][row]
  int n_sorted;
  int sorted[kMaxSortedHeads];
  int lens[kMaxSortedHeads];
  uint64_t pv_last;  // short K/V: an item's last PV product has been issued
};

struct Item {
  int b, h, kvh, q0, L;
  int j0;     // first K/V tile
  int n;      // K/V tiles the item visits: j0 .. j0 + n - 1
  int split;  // key range of a split-KV item (0 otherwise)
};

// The item of this CTA's pass `pass`: the persistent CTAs take the items in a snake order
// (CTA c takes c, 2G - 1 - c, 2G + c, ...), so that over a longest-first list (causal
// query blocks) the CTA that took a pass's longest item takes the next pass's shortest.
// Each pass still covers one contiguous block of items, as a plain round robin does.
__device__ __forceinline__ int item_at(int pass) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return (pass & 1) ? (pass + 1) * G - 1 - c : pass * G + c;
}

// This CTA's item after `idx`, its pass `pass`: the snake order, except for the paged kind,
// which goes round robin (its kernel compiled with the snake step ran the DiT
// self-attention 7 % slower, whatever the order it took).
template <int KIND>
__device__ __forceinline__ int next_item(int idx, int pass) {
  if constexpr (KIND == kPaged) return idx + static_cast<int>(gridDim.x);
  else return item_at(pass);
}

__device__ __forceinline__ int clamp_len(int L, int Skv) { return L < 0 ? 0 : (L > Skv ? Skv : L); }

__device__ __forceinline__ int len_at(const FwdParams& p, int b, int kvh) {
  return __ldg(p.kv_lens + b * p.lens_bstride + kvh * p.lens_hstride);
}

template <int KIND, typename Ctl>
__device__ __forceinline__ Item decode_item(int idx, const FwdParams& p, const Ctl& c) {
  const int g = p.fd_g.d;
  int split = 0;
  if (KIND == kSplit) {
    // the key range varies slowest: the CTAs running at the same time read the same keys
    // of all heads, whole rows of the [B, S, H, D] cache, rather than each its own 256-byte
    // pieces 10 KB apart (64 query rows over a 40-head, 32760-key cache: 134 -> 130 us)
    split = p.fd_range.div(idx);
    idx -= split * p.fd_range.d;
  }
  int b, h, qb;
  if (p.causal) {
    // longest first: the last query blocks see the most keys
    const int r = p.fd_bh.div(idx);
    qb = p.n_qblocks - 1 - r;
    const int bh = idx - r * p.fd_bh.d;
    b = p.fd_hq.div(bh);
    h = bh - b * p.Hq;
  } else if (c.n_sorted > 0) {
    // varlen: (batch, kv head) groups in decreasing valid length
    const int gi = p.fd_per.div(idx);
    const int bk = c.sorted[gi];
    const int rem = idx - gi * p.fd_per.d;
    b = p.fd_hkv.div(bk);
    const int hb = p.fd_qb.div(rem);
    h = (bk - b * p.Hkv) * g + hb;
    qb = rem - hb * p.n_qblocks;
  } else if (p.head_inner) {
    // short K/V (L2-resident): concurrent CTAs cover every head of the same query rows,
    // so Q is read and O written as whole contiguous rows across heads
    qb = p.fd_bh.div(idx);
    const int bh = idx - qb * p.fd_bh.d;
    b = p.fd_hq.div(bh);
    h = bh - b * p.Hq;
  } else {
    // long K/V: consecutive query blocks of one head run together and share K/V in L2
    const int bh = p.fd_qb.div(idx);
    qb = idx - bh * p.n_qblocks;
    b = p.fd_hq.div(bh);
    h = bh - b * p.Hq;
  }
  Item it;
  it.b = b;
  it.h = h;
  it.kvh = p.fd_g.div(h);
  it.q0 = qb * kItemRows;
  it.L = p.kv_lens ? clamp_len(len_at(p, b, it.kvh), p.Skv) : p.Skv;
  int kmax = it.L;
  if (p.causal) {
    const int ilast = min(it.q0 + kBM - 1, p.Sq - 1);
    kmax = min(it.L, ilast + it.L - p.Sq + 1);
  }
  kmax = max(kmax, 0);
  const int tiles = (kmax + kBN - 1) / kBN;
  it.split = split;
  it.j0 = KIND == kSplit ? split * p.split_tiles : 0;
  it.n = KIND == kSplit ? max(0, min(p.split_tiles, tiles - it.j0)) : tiles;
  return it;
}

// Whether K/V tile j holds in-bounds rows at or past the valid length (padding that may
// hold anything, even NaN): such a V tile gets the padding rows that the PV product reads
// zeroed before it.
__device__ __forceinline__ bool needs_fix(int j, int L, int Skv) {
  return min(Skv, (j + 1) * kBN) > L;
}

// Number of 16-key steps of the PV product for tile j: only steps holding valid keys.
__device__ __forceinline__ int pv_steps(int j, int L) {
  const int valid = min(kBN, L - j * kBN);
  return (valid + 15) / 16;
}

template <int D, int NQ, int NK, int NV, int KIND>
__global__ void __launch_bounds__(kThreads, 1) fwd_sm103_kernel(const __grid_constant__ FwdParams p) {
  constexpr int kQTile = kBM * D * 2;     // bytes of a Q tile
  constexpr int kKVTile = kBN * D * 2;    // bytes of a K or V tile
  constexpr int kQChunk = kBM * 128;      // 64 columns (128 bytes) of a Q tile
  constexpr int kKVChunk = kBN * 128;
  constexpr int kChunks = D / 64;
  constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, false, true);
  // TMEM columns: S double buffer [0, 256), P double buffer [256, 384) (bf16 pairs),
  // O [384, 384 + D); tile g uses S and P buffer g % 2
  constexpr uint32_t kColP = 256, kColO = 384;
  using Ctl = FwdCtl<NQ, NK, NV>;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                    // NQ tile slots
  uint8_t* sK = smem + NQ * kQTile;      // NK tile slots
  uint8_t* sV = sK + NK * kKVTile;       // NV tile slots
  uint8_t* sO = sV + NV * kKVTile;       // O staging tile (SW128 layout, as Q)
  Ctl& c = *reinterpret_cast<Ctl*>(sO + kQTile);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // split-KV: the merge that follows is a programmatic dependent of this grid (it waits
  // for this grid's completion before reading the partials), so its launch overlaps
  if (KIND == kSplit) griddep_launch_dependents();

  // ------------------------------------------------------------------- prologue
  if (threadIdx.x == 0) {
    mbar_init(&c.mma_final[0], 1);
    mbar_init(&c.mma_final[1], 1);
    for (int s = 0; s < NQ; ++s) {
      mbar_init(&c.q_full[s], 1);
      mbar_init(&c.q_empty[s], 1);
    }
    for (int s = 0; s < NK; ++s) {
      mbar_init(&c.k_full[s], 1);
      mbar_init(&c.k_empty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&c.v_full[s], 1);
      mbar_init(&c.v_empty[s], 1);
      mbar_init(&c.v_fixed[s], 1);
      mbar_init(&c.fix_req[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&c.s_full[b], 1);
      mbar_init(&c.s_free[b], kSoftThreads);
      mbar_init(&c.pv_done[b], 1);
      mbar_init(&c.p_full[b], kSoftThreads);
    }
    mbar_init(&c.o_free, kSoftThreads);
    if (NQ == 1) mbar_init(&c.pv_last, 1);  // used by the short-K/V configuration only
    for (int q = 0; q < 4; ++q) {
      mbar_init(&c.xfull[q], 64);
      mbar_init(&c.xdone[q], 64);
    }
    mbar_init(&c.o_staged, kSoftThreads);
    mbar_init(&c.stage_free, 1);
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
      const int raw = len_at(p, e / p.Hkv, e % p.Hkv);
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
  // Registers: the control warpgroup (warps 0-3) gives 16 of its 168 to each thread of
  // the two softmax warpgroups (measured: cross-attention 533 -> 544 TFLOP/s, DiT self
  // within noise; 136 / 184 was slower). The paged kernel keeps the plain allocation (the
  // split cost it 5 %: its producer's page lookups need the registers). The split adds up
  // to exactly the registers the block is launched with (384 x 168), which launch()
  // checks before the first launch.
  static_assert(4 * 32 * kRegsCtl + 8 * 32 * kRegsSoft == kThreads * kRegsLaunch, "register split");
  if constexpr (KIND != kPaged) {
    if (warp < 4)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
    else
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoft));
  }

  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_map(&p.tm_q);
      tma_prefetch_map(&p.tm_k);
      tma_prefetch_map(&p.tm_v);
    }
    // Paged K/V: block-table entries are read 32 at a time, one per lane, and handed out
    // by shuffles, so the producer does not wait for a global load before every tile. One
    // cache for K and one for V (K runs ahead of V); reset at every item.
    struct PageCache {
      int base, val;
    };
    PageCache pc_k{-1, 0}, pc_v{-1, 0};
    auto page_of = [&](PageCache& pc, int b, int e) -> int {  // warp-uniform e
      if (pc.base < 0 || e < pc.base || e >= pc.base + 32) {
        pc.base = e;
        pc.val = e + lane < p.max_pages ? __ldg(p.block_table + (int64_t)b * p.max_pages + e + lane) : 0;
      }
      return __shfl_sync(0xffffffffu, pc.val, e - pc.base);
    };
    // K/V tile jj of an item into `dst`, completing on `bar`; called by the whole warp,
    // lane 0 issues. Dense: one box of 128 keys per 64-column chunk. Paged: the tile's keys
    // in boxes of page_box rows, each inside one page; boxes that start at or past the
    // valid length are not loaded (their keys are masked, and the V rows that the PV
    // product reads there are zeroed by warp 2).
    auto load_kv = [&](uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int jj, const Item& it,
                       PageCache& pc) {
      if constexpr (KIND != kPaged) {
        if (lane == 0) {
          mbar_expect_tx(bar, kKVTile);
          for (int ch = 0; ch < kChunks; ++ch)
            tma_load_4d(dst + ch * kKVChunk, map, bar, ch * 64, it.kvh, jj * kBN, it.b);
        }
      } else {
        const int valid = min(kBN, it.L - jj * kBN);  // >= 1: tile jj holds valid keys
        const int box = 1 << p.box_shift;
        const int boxes = (valid + box - 1) >> p.box_shift;
        if (lane == 0) mbar_expect_tx(bar, (uint32_t)(boxes << p.box_shift) * 128 * kChunks);
        for (int x = 0; x < boxes; ++x) {
          const int t0 = jj * kBN + (x << p.box_shift);
          int page = page_of(pc, it.b, t0 >> p.page_shift);
          if (lane == 0) {
            if (page < 0 || page >= p.num_pages) {
              atomicOr(p.err, ATTN_DEVERR_PAGE);
              page = 0;  // a page that exists: the call's outputs are invalid, nothing faults
            }
            for (int ch = 0; ch < kChunks; ++ch)
              tma_load_4d(dst + ch * kKVChunk + (x << p.box_shift) * 128, map, bar, ch * 64, it.kvh,
                          t0 & ((1 << p.page_shift) - 1), page);
          }
        }
      }
    };
    // K_j is read by S(j), which runs up to two tiles ahead of PV(j); so K is loaded two
    // tiles ahead of V and kept on its own ring, freed as soon as S(j) completes
    uint32_t kpos = 0, vpos = 0, qs = 0, q_par = 0;
    uint32_t k_iss = 0, k_last = 0, v_iss = 0, v_last = 0;  // per slot: a load was issued / its parity
    uint32_t q_issued = 0, q_last = 0;                      // per Q slot
    bool ok = true, first = true;
    for (int ps = 0, idx = item_at(0); ok && idx < p.n_items; idx = next_item<KIND>(idx, ++ps)) {
      const Item it = decode_item<KIND>(idx, p, c);
      if (it.n == 0) continue;
      pc_k.base = -1;  // a new sequence: its block-table row
      pc_v.base = -1;
      if (!wait_phase_warp(&c.q_empty[qs], q_par ^ 1, wc)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(&c.q_full[qs], kQTile);
        for (int ch = 0; ch < kChunks; ++ch)
          tma_load_4d(sQ + qs * kQTile + ch * kQChunk, &p.tm_q, &c.q_full[qs], ch * 64, it.h, it.q0, it.b);
      }
      q_issued |= 1u << qs;
      q_last = (q_last & ~(1u << qs)) | (q_par << qs);
      if (++qs == NQ) { qs = 0; q_par ^= 1; }
      for (int step = 0; ok && step < it.n + 2; ++step) {
        if (step < it.n) {
          const int j = step;
          const uint32_t ks = kpos % NK, kpar = (kpos / NK) & 1;
          if (!wait_phase_warp(&c.k_empty[ks], kpar ^ 1, wc)) { ok = false; break; }
          const bool skip = (p.fault & 1u) && blockIdx.x == 0 && first && j == 0;
          if (!skip) {
            load_kv(sK + ks * kKVTile, &p.tm_k, &c.k_full[ks], it.j0 + j, it, pc_k);
            k_iss |= 1u << ks;
            k_last = (k_last & ~(1u << ks)) | (kpar << ks);
          }
          ++kpos;
        }
        if (step >= 2) {
          const int j = step - 2;
          const uint32_t vs = vpos % NV, vpar = (vpos / NV) & 1;
          if (!wait_phase_warp(&c.v_empty[vs], vpar ^ 1, wc)) { ok = false; break; }
          load_kv(sV + vs * kKVTile, &p.tm_v, &c.v_full[vs], it.j0 + j, it, pc_v);
          v_iss |= 1u << vs;
          v_last = (v_last & ~(1u << vs)) | (vpar << vs);
          // a V tile with padding rows: warp 2 zeroes them once the tile has landed
          if (needs_fix(it.j0 + j, it.L, p.Skv) && lane == 0) mbar_arrive(&c.fix_req[vs]);
          ++vpos;
        }
      }
      first = false;
    }
    // every copy this CTA started lands before its shared memory can go away (after an
    // abort the consumers may never have waited for them)
    for (int s = 0; s < NK; ++s)
      if (k_iss & (1u << s)) wait_phase_teardown(&c.k_full[s], (k_last >> s) & 1, 200000000ull);
    for (int s = 0; s < NV; ++s)
      if (v_iss & (1u << s)) wait_phase_teardown(&c.v_full[s], (v_last >> s) & 1, 200000000ull);
    for (int s = 0; s < NQ; ++s)
      if (q_issued & (1u << s)) wait_phase_teardown(&c.q_full[s], (q_last >> s) & 1, 200000000ull);
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------- MMA issuers
    // S(j) goes to S buffer j % 2 as soon as the softmax has read S(j - 2) out of it, so
    // the S product of a later tile always runs while the softmax works on the current
    // one; PV(j) follows once P(j) is written into P buffer j % 2. P has its own
    // columns, so no S product ever waits for a PV product.
    // warp 1 issues the S products, warp 3 the PV products: each thread's waits then
    // block only its own product family (a wait costs hundreds of cycles while SS MMAs
    // hold the shared-memory bandwidth)
    const bool s_role = warp == 1;
    if (lane == 0) {
      const uint32_t sQa = smem_u32(sQ);
      // K-major Q and K tiles (128-byte rows, 8-row groups 1024 bytes apart); MN-major V
      // (64-column chunks kKVChunk bytes apart)
      const uint64_t desc_q0 = smem_desc_sw128(sQa, 16, 1024);
      const uint64_t desc_k0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t desc_v0 = smem_desc_sw128(smem_u32(sV), kKVChunk, 1024);
      // ring positions: the k-th loaded item's Q tile is Q position k; its K and V tiles j
      // are at position kbase + j of the K and the V ring; a position's slot is pos % N and
      // its phase parity (pos / N) % 2
      uint32_t kbase = 0, qpos = 0, fix_par = 0, gs = 0, gp = 0, ic = 0;
      bool ok = true;
      auto issue_s = [&](uint32_t qslot, int j) -> bool {
        const uint32_t kpos = kbase + j, ks = kpos % NK;
        if (!wait_phase(&c.k_full[ks], (kpos / NK) & 1, wc)) return false;
        const uint32_t b = gs & 1;
        if (gs >= 2 && !wait_phase(&c.s_free[b], ((gs >> 1) - 1) & 1, wc)) return false;
        tc_fence_after();
        const uint64_t a0 = desc_q0 + ((qslot * kQTile) >> 4);
        const uint64_t b0 = desc_k0 + ((ks * kKVTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + b * 128, a0 + (((kk / 4) * kQChunk + (kk % 4) * 32) >> 4),
                 b0 + (((kk / 4) * kKVChunk + (kk % 4) * 32) >> 4), kIdescS, kk > 0 ? 1u : 0u);
        mma_commit(&c.s_full[b]);
        mma_commit(&c.k_empty[ks]);  // K_j is read by this product only
        ++gs;
        return true;
      };
      // PV of the item's tile j (local index), key tile jj = j0 + j of the sequence
      auto issue_pv = [&](int j, int jj, int L) -> bool {
        const uint32_t vpos = kbase + j, vs = vpos % NV;
        if (needs_fix(jj, L, p.Skv)) {
          if (!wait_phase(&c.v_fixed[vs], (fix_par >> vs) & 1, wc)) return false;
          fix_par ^= 1u << vs;
        } else if (!wait_phase(&c.v_full[vs], (vpos / NV) & 1, wc)) {
          return false;
        }
        if (!wait_phase(&c.p_full[gp & 1], (gp >> 1) & 1, wc)) return false;
        if (j == 0 && !wait_phase(&c.o_free, (ic & 1) ^ 1, wc)) return false;
        tc_fence_after();
        const int steps = pv_steps(jj, L);
        const uint64_t b0 = desc_v0 + ((vs * kKVTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          if (kk < steps)
            mma_ts(tmem + kColO, tmem + kColP + (gp & 1) * 64 + kk * 8, b0 + ((kk * 16 * 128) >> 4), kIdescPV,
                   (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&c.pv_done[gp & 1]);
        mma_commit(&c.v_empty[vs]);
        ++gp;
        return true;
      };
      for (int ps = 0, idx = item_at(0); ok && idx < p.n_items; idx = next_item<KIND>(idx, ++ps)) {
        const Item it = decode_item<KIND>(idx, p, c);
        if (it.n == 0) continue;
        const uint32_t qslot = qpos % NQ;
        if (s_role && !wait_phase(&c.q_full[qslot], (qpos / NQ) & 1, wc)) { ok = false; break; }
        ++qpos;
        tc_fence_after();
        // Short K/V (one Q slot): the tensor pipe runs both issuers' products in one
        // order, and an item's last PV is on the way to its epilogue, so the next item's
        // first S waits until that PV has been issued (it then runs under the epilogue
        // rather than ahead of the PV).
        constexpr bool kPvFirst = NQ == 1;
        if (s_role) {
          if (kPvFirst && ic > 0 && !wait_phase(&c.pv_last, (ic - 1) & 1, wc)) { ok = false; break; }
          // S(t) as soon as its K tile is in and the softmax has read S(t - 2)
          for (int t = 0; ok && t < it.n; ++t) ok = issue_s(qslot, t);
          if (!ok) break;
          mma_commit(&c.q_empty[qslot]);  // last read of Q
        } else {
          // PV(t) once the softmax has written P(t)
          for (int t = 0; ok && t < it.n; ++t) ok = issue_pv(t, it.j0 + t, it.L);
          if (!ok) break;
          if (kPvFirst) mbar_arrive(&c.pv_last);
        }
        kbase += it.n;
        ++ic;
      }
      // every MMA this thread issued must finish before the TMEM is freed
      mma_commit(&c.mma_final[s_role ? 0 : 1]);
      wait_phase_teardown(&c.mma_final[s_role ? 0 : 1], 0, 200000000ull);
    }
    __syncwarp();
  } else if (warp == 2) {
    // -------------------------------------------------------------- V-tile fixer
    // zeroes the padding rows (at or past the valid length) of partial V tiles, so
    // that 0 * NaN in the PV product cannot occur; requests come from the producer
    // in ring order (fix_req), so the fill this waits for is never ambiguous
    uint32_t kbase = 0, fr_par = 0;
    bool ok = true;
    for (int ps = 0, idx = item_at(0); ok && idx < p.n_items; idx = next_item<KIND>(idx, ++ps)) {
      const Item it = decode_item<KIND>(idx, p, c);
      if (it.n == 0) continue;
      for (int j = 0; j < it.n; ++j) {
        const int jj = it.j0 + j;
        if (!needs_fix(jj, it.L, p.Skv)) continue;
        const uint32_t vpos = kbase + j, vs = vpos % NV;
        if (!wait_phase_warp(&c.fix_req[vs], (fr_par >> vs) & 1, wc)) { ok = false; break; }
        fr_par ^= 1u << vs;
        if (!wait_phase_warp(&c.v_full[vs], (vpos / NV) & 1, wc)) { ok = false; break; }
        const int r0 = it.L - jj * kBN;  // first padding row (>= 1: tile jj holds valid keys)
        // the PV product reads whole 16-key steps up to the last valid key: only padding
        // rows inside that last step are read, and only they are zeroed
        const int r1 = pv_steps(jj, it.L) * 16;
        const int units = (r1 - r0) * kChunks * 8;
        uint8_t* base = sV + vs * kKVTile;
        for (int e = lane; e < units; e += 32) {
          const int r = r0 + e / (kChunks * 8);
          const int rest = e % (kChunks * 8);
          *reinterpret_cast<uint4*>(base + (rest / 8) * kKVChunk + r * 128 + (rest % 8) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.v_fixed[vs]);
      }
      kbase += it.n;
    }
  } else if (warp >= 4) {
    // --------------------------------------------------------------------- softmax
    // Two threads per row: warp w reaches TMEM lanes 32 * (w % 4) .. and takes the key
    // columns 64 h .. 64 h + 63 of each tile, h = (w - 4) / 4. The pair trades its
    // partial row max every tile (and its partial row sum at the end) through shared
    // memory, so both halves use the same running max; each half keeps its own part of
    // the row sum and rescales its half of O.
    const int quad = warp % 4;
    const int h = (warp - 4) / 4;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tO = tmem + lane_off + kColO + h * (D / 2);
    const bool pos_scale = p.scale_log2 > 0.f;
    uint32_t g = 0;   // tiles processed so far (all items): S and P buffer g % 2, PV number g
    uint32_t xc = 0;  // exchanges with the other half of the row so far
    uint32_t ic_s = 0;  // items with tiles finished (O staging tile uses)
    bool ok = true;
    // hands `v` to the other half of the row and returns its value
    auto trade = [&](float v, float& other) -> bool {
      if (xc > 0 && !wait_phase_warp(&c.xdone[quad], (xc - 1) & 1, wc)) return false;
      c.xbuf[h][r] = v;
      mbar_arrive(&c.xfull[quad]);
      if (!wait_phase_warp(&c.xfull[quad], xc & 1, wc)) return false;
      other = c.xbuf[1 - h][r];
      mbar_arrive(&c.xdone[quad]);
      ++xc;
      return true;
    };
    for (int ps = 0, idx = item_at(0); ok && idx < p.n_items; idx = next_item<KIND>(idx, ++ps)) {
      const Item it = decode_item<KIND>(idx, p, c);
      const int i = it.q0 + r;
      const bool row_ok = i < p.Sq;
      __nv_bfloat16* orow = p.o + ((static_cast<int64_t>(it.b) * p.Sq + i) * p.Hq + it.h) * D + h * (D / 2);
      float* lrow = p.lse + (static_cast<int64_t>(it.b) * p.Hq + it.h) * p.Sq + i;
      // split-KV items write their normalised partial O and LSE (fp32) instead
      const int64_t prow = ((static_cast<int64_t>(it.split) * p.B + it.b) * p.Hq + it.h) * p.Sq + i;
      float* porow = KIND == kSplit ? p.o_part + prow * D + h * (D / 2) : nullptr;
      if (it.n == 0) {
        if (row_ok) {
          if (KIND == kSplit) {
            for (int d = 0; d < D / 2; d += 4)
              *reinterpret_cast<float4*>(porow + d) = make_float4(0.f, 0.f, 0.f, 0.f);
            if (h == 0) p.lse_part[prow] = -CUDART_INF_F;
          } else {
            for (int d = 0; d < D / 2; d += 8)
              *reinterpret_cast<uint4*>(orow + d) = make_uint4(0u, 0u, 0u, 0u);
            if (h == 0) *lrow = -CUDART_INF_F;
          }
        }
        continue;
      }
      // visible keys of this row: [0, kend)
      const int kend = p.causal ? min(it.L, i + it.L - p.Sq + 1) : it.L;
      float m = -CUDART_INF_F, l = 0.f;
      for (int j = 0; j < it.n; ++j, ++g) {
        const uint32_t b = g & 1;
        if (!wait_phase_warp(&c.s_full[b], (g >> 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        // visible columns of this half: e < limit
        const int limit = kend - (it.j0 + j) * kBN - 64 * h;
        // one TMEM round trip: this half of the S row into registers, which (with the
        // other half) frees the buffer for S(j + 2)
        float s[64];
        tmem_ld64(tmem + lane_off + b * 128 + 64 * h, reinterpret_cast<uint32_t*>(s));
        tc_fence_before();
        mbar_arrive(&c.s_free[b]);
        // the half row max, 8 independent chains; for a positive scale the max of the raw
        // scores, scaled once
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = -CUDART_INF_F;
        const bool full = limit >= 64;
        if (pos_scale && full) {
#pragma unroll
          for (int e = 0; e < 32; ++e) mx8[e % 8] = max3f(mx8[e % 8], s[2 * e], s[2 * e + 1]);
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) {
            const float v = pos_scale ? s[e] : s[e] * p.scale_log2;
            mx8[e % 8] = fmaxf(mx8[e % 8], e < limit ? v : -CUDART_INF_F);
          }
        }
        const float mxh = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        float mxo;
        if (!trade(mxh, mxo)) { ok = false; break; }
        const float mx = fmaxf(mxh, mxo);  // the same value in both halves
        const float mnew = fmaxf(m, pos_scale ? mx * p.scale_log2 : mx);
        const bool raise = mnew > m + kRescaleThreshold;
        const bool rescale = raise && m != -CUDART_INF_F;
        // TMEM loads/stores are warp-collective: the warp rescales together, rows that
        // need no rescale with a factor of 1. O holds the sum through PV(g - 1) once that
        // product completes (rescale implies j > 0).
        if (__any_sync(0xffffffffu, rescale)) {
          if (!wait_phase_warp(&c.pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          const float alpha = rescale ? ex2_approx(m - mnew) : 1.f;
          l *= alpha;
#pragma unroll 1
          for (int cc = 0; cc < D / 64; ++cc) {
            uint32_t ov[32];
            tmem_ld32(tO + cc * 32, ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(tO + cc * 32, ov);
          }
        }
        if (raise) m = mnew;
        // P = 2^(s * scale * log2 e - m) in bf16 into P buffer g % 2 (this half's 32
        // columns), in two quarters; the first store waits until PV(g - 2) has read that
        // buffer
        const float msub = m == -CUDART_INF_F ? 0.f : m;
        const uint32_t tP = tmem + lane_off + kColP + b * 64 + 32 * h;
        float rs8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) rs8[e] = 0.f;
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          uint32_t pk[16];
          if (q2 > 0) reg_fence32(s + q2 * 32);  // after the previous quarter's store
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c0 = q2 * 32 + 2 * e;
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
          if (q2 == 0 && g >= 2) {
            if (!wait_phase_warp(&c.pv_done[b], ((g >> 1) - 1) & 1, wc)) { ok = false; break; }
            tc_fence_after();
          }
          tmem_st16(tP + q2 * 16, pk);
        }
        if (!ok) break;
        l += ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&c.p_full[b]);
      }
      if (!ok) break;
      // epilogue: the row sum of both halves (added in a fixed order), then O / l and
      // LSE once PV(g - 1), the item's last, has completed
      float lo;
      if (!trade(l, lo)) { ok = false; break; }
      const float lt = h == 0 ? l + lo : lo + l;
      if (!wait_phase_warp(&c.pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, wc)) { ok = false; break; }
      tc_fence_after();
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float lse_nat = lt > 0.f ? (m + __log2f(lt)) * 0.69314718055994531f : -CUDART_INF_F;
      if (KIND == kSplit) {
        // a split-KV partial: this half row of O / l in fp32 (32-byte stores, the row is
        // contiguous and 512-byte aligned), then its LSE; fwd_combine_kernel merges them
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          uint32_t ov[32];
          tmem_ld32(tO + cc * 32, ov);
          if (row_ok) {
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * inv);
#pragma unroll
            for (int e = 0; e < 4; ++e) st_global_v8(porow + cc * 32 + e * 8, ov + 8 * e);
          }
        }
        tc_fence_before();
        mbar_arrive(&c.o_free);
        if (row_ok && h == 0) p.lse_part[prow] = lse_nat;
        continue;
      }
      // O goes out through shared memory and TMA tile stores: written straight from the
      // registers, each thread's row slice would be 16-byte stores 32 rows apart. The
      // staging tile is free once the previous item's store has read it.
      // Warp 4 issued the previous item's store and confirms here, an item later, that it
      // has read the tile, so no softmax warp waits for the store at the end of an item.
      if (warp == 4 && lane == 0 && ic_s > 0) {
        tma_store_wait_read();
        mbar_arrive(&c.stage_free);
      }
      if (!wait_phase_warp(&c.stage_free, (ic_s & 1) ^ 1, wc)) { ok = false; break; }
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t ov[32];
        tmem_ld32(tO + cc * 32, ov);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          // columns col .. col + 7: 64-column chunk col / 64, 16-byte unit of its 128-byte
          // row (col % 64) / 8, placed with the 128-byte swizzle of the tensor map
          const int col = h * (D / 2) + cc * 32 + e * 8;
          const int u = (col & 63) >> 3;
          *reinterpret_cast<uint4*>(sO + (col >> 6) * (kBM * 128) + r * 128 + ((u ^ (r & 7)) * 16)) =
              make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&c.o_free);  // O's columns may be overwritten
      fence_proxy_async_smem();
      mbar_arrive(&c.o_staged);
      if (row_ok && h == 0) *lrow = lse_nat;
      if (warp == 4) {
        if (!wait_phase_warp(&c.o_staged, ic_s & 1, wc)) { ok = false; break; }
        if (lane == 0) {
#pragma unroll
          for (int ch = 0; ch < D / 64; ++ch) tma_store_4d(&p.tm_o, sO + ch * (kBM * 128), ch * 64, it.h, it.q0, it.b);
          tma_store_commit();
        }
        __syncwarp();
      }
      ++ic_s;
    }
    // the last stores complete before the CTA exits
    if (warp == 4 && lane == 0) tma_store_wait_all();
  }

  // ---------------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// The merge of split-KV partials: one warp per query row (b, h, i). With lse_s and O_s
// the partial LSE and normalised output of key range s (lse_s = -inf for a range with no
// visible key), lse = m + log(sum_s exp(lse_s - m)), m = max_s lse_s, and
// O = sum_s exp(lse_s - lse) O_s, summed in range order (deterministic); a row with no
// visible key at all gets O = 0, lse = -inf. Launched as a programmatic dependent of the
// forward grid.
template <int D>
__global__ void __launch_bounds__(256) fwd_combine_kernel(const float* __restrict__ o_part,
                                                          const float* __restrict__ lse_part,
                                                          __nv_bfloat16* __restrict__ o,
                                                          float* __restrict__ lse, int B, int Hq,
                                                          int Sq, int n_splits) {
  constexpr int kPer = D / 32;  // columns per lane
  griddep_wait();
  const int64_t rows = (int64_t)B * Hq * Sq;
  const int64_t row = (int64_t)blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  float m = -CUDART_INF_F;
  for (int sp = lane; sp < n_splits; sp += 32) m = fmaxf(m, lse_part[sp * rows + row]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (m != -CUDART_INF_F) {
    for (int sp = 0; sp < n_splits; ++sp) {
      const float ls = lse_part[sp * rows + row];
      if (ls == -CUDART_INF_F) continue;
      const float wgt = expf(ls - m);
      wsum += wgt;
      const float* src = o_part + (sp * rows + row) * D + lane * kPer;
      if constexpr (kPer == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        acc[0] += wgt * x.x; acc[1] += wgt * x.y; acc[2] += wgt * x.z; acc[3] += wgt * x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        acc[0] += wgt * x.x; acc[1] += wgt * x.y;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int i = (int)(row % Sq);
  const int64_t bh = row / Sq;
  const int h = (int)(bh % Hq), b = (int)(bh / Hq);
  __nv_bfloat16* dst = o + (((int64_t)b * Sq + i) * Hq + h) * D + lane * kPer;
  uint32_t pk[kPer / 2];
#pragma unroll
  for (int e = 0; e < kPer / 2; ++e) pk[e] = pack_bf16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
  if constexpr (kPer == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pk[0];
  }
  if (lane == 0) lse[row] = wsum > 0.f ? m + logf(wsum) : -CUDART_INF_F;
}

// ---------------------------------------------------------------------- host side
template <int D, int NQ, int NK, int NV>
constexpr size_t fwd_smem_bytes() {
  return 1024 + (size_t)(NQ + 1) * kBM * D * 2 + (size_t)(NK + NV) * kBN * D * 2 + sizeof(FwdCtl<NQ, NK, NV>);
}

constexpr int kMaxDev = 64;
std::mutex g_mu;
int g_num_sms[kMaxDev] = {};

template <int D, int NQ, int NK, int NV, int KIND>
cudaError_t launch(const FwdParams& prm, int dev, cudaStream_t s) {
  constexpr size_t smem = fwd_smem_bytes<D, NQ, NK, NV>();
  static_assert(smem <= 232448, "shared memory per block");
  {
    // the shared-memory opt-in, once per kernel instantiation and device
    static bool attr_set[kMaxDev] = {};
    std::lock_guard<std::mutex> lk(g_mu);
    if (!attr_set[dev]) {
      // the register split inside the kernel assumes exactly kRegsLaunch registers a
      // thread at launch; with fewer the softmax warps' increase could never be granted
      cudaFuncAttributes fa{};
      cudaError_t ea = cudaFuncGetAttributes(&fa, fwd_sm103_kernel<D, NQ, NK, NV, KIND>);
      if (ea != cudaSuccess) return ea;
      if (KIND != kPaged && fa.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
      cudaError_t e = cudaFuncSetAttribute(fwd_sm103_kernel<D, NQ, NK, NV, KIND>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
  }
  const int grid = prm.n_items < g_num_sms[dev] ? prm.n_items : g_num_sms[dev];
  fwd_sm103_kernel<D, NQ, NK, NV, KIND><<<grid, kThreads, smem, s>>>(prm);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || KIND != kSplit) return e;
  const int64_t rows = (int64_t)prm.B * prm.Hq * prm.Sq;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)((rows + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, fwd_combine_kernel<D>, static_cast<const float*>(prm.o_part),
                         static_cast<const float*>(prm.lse_part), prm.o, prm.lse, prm.B, prm.Hq,
                         prm.Sq, prm.n_splits);
  if (e != cudaSuccess) return e;
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

// A bf16 page pool [num_pages, page_size, H, D] as a 4-D TMA map (D, H, page_size,
// num_pages) whose box is one head: 64 columns (128 bytes, 128-byte swizzle) x `rows`
// keys of one page.
bool make_page_map(CUtensorMap* map, const void* base, int num_pages, int page_size, int H, int D,
                   int rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)page_size,
                              (cuuint64_t)num_pages};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2,
                                 (cuuint64_t)page_size * H * D * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
  const bool paged = p.block_table != nullptr;
  // with no keys the K/V maps are never used; describe q so that encoding succeeds
  const bool no_keys = p.Skv == 0;
  bool maps_ok = make_bshd_map(&prm.tm_q, p.q, p.B, p.Sq, p.Hq, p.D, kBM) &&
                 make_bshd_map(&prm.tm_o, p.o, p.B, p.Sq, p.Hq, p.D, kBM);
  if (paged && !no_keys) {
    const int box = p.page_size < kBN ? p.page_size : kBN;
    maps_ok = maps_ok && make_page_map(&prm.tm_k, p.k, p.num_pages, p.page_size, p.Hkv, p.D, box) &&
              make_page_map(&prm.tm_v, p.v, p.num_pages, p.page_size, p.Hkv, p.D, box);
    while ((1 << prm.page_shift) < p.page_size) ++prm.page_shift;
    while ((1 << prm.box_shift) < box) ++prm.box_shift;
  } else {
    maps_ok = maps_ok &&
              make_bshd_map(&prm.tm_k, no_keys ? p.q : p.k, p.B, no_keys ? p.Sq : p.Skv,
                            no_keys ? p.Hq : p.Hkv, p.D, kBN) &&
              make_bshd_map(&prm.tm_v, no_keys ? p.q : p.v, p.B, no_keys ? p.Sq : p.Skv,
                            no_keys ? p.Hq : p.Hkv, p.D, kBN);
  }
  if (!maps_ok) return cudaErrorInvalidValue;
  prm.o = static_cast<__nv_bfloat16*>(p.o);
  prm.lse = p.lse;
  prm.kv_lens = p.kv_lens;
  // a paged cache has one valid length per sequence, shared by its kv heads
  prm.lens_bstride = paged ? 1 : p.Hkv;
  prm.lens_hstride = paged ? 0 : 1;
  prm.block_table = paged ? p.block_table : nullptr;
  prm.max_pages = p.max_pages;
  prm.num_pages = p.num_pages;
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
  prm.n_splits = p.fwd_splits > 1 ? p.fwd_splits : 1;
  prm.split_tiles = p.fwd_split_tiles;
  prm.o_part = p.o_part;
  prm.lse_part = p.lse_part;
  prm.n_items = p.B * p.Hq * prm.n_qblocks * prm.n_splits;
  const int g = p.Hq / p.Hkv;
  prm.fd_range = FastDiv::make(p.B * p.Hq * prm.n_qblocks);
  prm.fd_bh = FastDiv::make(p.B * p.Hq);
  prm.fd_hq = FastDiv::make(p.Hq);
  prm.fd_hkv = FastDiv::make(p.Hkv);
  prm.fd_qb = FastDiv::make(prm.n_qblocks);
  prm.fd_g = FastDiv::make(g);
  prm.fd_per = FastDiv::make(g * prm.n_qblocks);
  prm.scale_log2 = p.scale * 1.4426950408889634f;
  prm.timeout_ns = 4000000000ull;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    prm.fault = g_fault_next;
    if (g_fault_next != 0 && g_fault_timeout_ns != 0) prm.timeout_ns = g_fault_timeout_ns;
    g_fault_next = 0;
  }
  const int kind = paged ? kPaged : (prm.n_splits > 1 ? kSplit : kDense);
  if (p.D == 64) {
    if (kind == kPaged) return launch<64, 3, 5, 4, kPaged>(prm, dev, s);
    if (kind == kSplit) return launch<64, 3, 5, 4, kSplit>(prm, dev, s);
    return launch<64, 3, 5, 4, kDense>(prm, dev, s);
  }
  if (kind == kPaged) return launch<128, 2, 2, 2, kPaged>(prm, dev, s);
  if (kind == kSplit) return launch<128, 2, 2, 2, kSplit>(prm, dev, s);
  // short K/V (items of at most 16 tiles: cross-attention to text tokens, 2k-token
  // training): one Q slot and three K slots, so that a K load of the next item does not
  // wait for this item's first S (DiT cross-attention 498 -> 514 TFLOP/s, GQA profiling
  // shape 880 -> 892; on long K/V the Q prefetch is worth more)
  if (p.Skv <= 16 * kBN) return launch<128, 1, 3, 2, kDense>(prm, dev, s);
  return launch<128, 2, 2, 2, kDense>(prm, dev, s);
}

}  // namespace attn
