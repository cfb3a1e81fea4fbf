"""Seeded synthetic workloads: shapes, value distributions and valid key lengths.

This module only draws random inputs. It holds no attention arithmetic, and it is the
one piece of code that both the CUDA path's tests/bench and the float64 oracle use, so
that both sides see the very same input values.

The workloads stand in for the real activations the pages profile (which are not
available here), with the pages' shapes:

* ``c1``  tiny MHA sanity: B1 H2 S128 D64, fp32, causal;
* ``c2``  decoder training shape: B8 H12 S1024 D64, bf16, causal (fwd + bwd);
* ``c3``  GQA training: B4 Hq8 Hkv2 S2048 D128, bf16, causal (query head h reads kv head
  h // 4; "xtrain evolution.md", table row T15);
* ``c4``  video-DiT self-attention, 21 frames x 30 x 52 latent patches = 32760 tokens,
  H40 D128, bf16, non-causal, Q and K scaled by 0.5 ("LingBot full-pipeline analysis
  report", section "Attention: real inputs, backends, errors and timing", self rows);
* ``c4v`` the same with per-head valid K/V lengths drawn uniformly from [1560, 32760]
  (the report's varlen FA3 path with cu_seqlens shorter than the allocation, section
  "same-GPU FA2/FA3 hardware comparison");
* ``c5``  video-DiT cross-attention: Sq 32760 video tokens, Skv 512 text tokens of which
  300 are valid (section "recorded cross-attention matrix work": K = 512 text tokens);
* ``vae_f32`` fp32 attention over one 60 x 104 latent frame (the report's fp32 VAE frame
  attention, fmha_cutlassF_f32), 8 heads of 128 (not stated on the pages).

Recipe: a CPU ``torch.Generator`` seeded with 20260 + the config number draws fp32
standard normals in the order Q, K, V, dO (dO only where the workload has a backward);
Q and K are multiplied by their factor; each tensor is then rounded to the workload's
dtype (round-to-nearest-even for bf16). Varlen lengths are drawn last, from the same
generator.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = ["Workload", "WORKLOADS", "get", "make_inputs", "small_case", "make_paged"]


@dataclass(frozen=True)
class Workload:
    key: str
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    D: int
    dtype: str  # "bf16" or "f32"
    causal: bool
    seed: int
    qk_factor: float = 1.0
    has_bwd: bool = False
    lens_kind: str = "none"  # "none" | "per_head_uniform" | "fixed"
    lens_lo: int = 0
    lens_hi: int = 0
    lens_fixed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def describe(self) -> str:
        return (f"{self.name}: B{self.B} Hq{self.Hq} Hkv{self.Hkv} Sq{self.Sq} Skv{self.Skv} "
                f"D{self.D} {self.dtype} {'causal' if self.causal else 'non-causal'}"
                + (f" lens={self.lens_kind}" if self.lens_kind != "none" else ""))


WORKLOADS = {
    "c1": Workload("c1", "tiny_mha_fp32_causal", 1, 2, 2, 128, 128, 64, "f32", True, 20261,
                   has_bwd=True),
    "c2": Workload("c2", "decoder_train_b8_h12_s1024_d64", 8, 12, 12, 1024, 1024, 64, "bf16",
                   True, 20262, has_bwd=True),
    "c3": Workload("c3", "gqa_train_b4_hq8_hkv2_s2048_d128", 4, 8, 2, 2048, 2048, 128, "bf16",
                   True, 20263, has_bwd=True),
    "c4": Workload("c4", "dit_self_s32760_h40_d128", 1, 40, 40, 32760, 32760, 128, "bf16",
                   False, 20264, qk_factor=0.5),
    "c4v": Workload("c4v", "dit_self_varlen_s32760_h40_d128", 1, 40, 40, 32760, 32760, 128,
                    "bf16", False, 20264, qk_factor=0.5, lens_kind="per_head_uniform",
                    lens_lo=1560, lens_hi=32760),
    "c5": Workload("c5", "dit_cross_sq32760_skv512_valid300_h40_d128", 1, 40, 40, 32760, 512,
                   128, "bf16", False, 20265, lens_kind="fixed", lens_fixed=300),
    # the report's own attention-timing shape (480 x 832 video, frame 27: 4680 queries over
    # a 28080-token KV cache, 40 heads): context for its FA3 figure, not a graded workload
    "ctx": Workload("ctx", "page_dit_self_q4680_k28080_h40_d128", 1, 40, 40, 4680, 28080, 128,
                    "bf16", False, 20268, qk_factor=0.5),
    # fp32 attention over one latent frame of the 480 x 832 video (60 x 104 = 6240
    # tokens), the role of the report's VAE frame attention (fmha_cutlassF_f32 in
    # vae_frame); the report gives neither its head count nor its head dimension, so 8
    # heads of 128 stand in
    "vae_f32": Workload("vae_f32", "vae_frame_f32_b1_h8_s6240_d128", 1, 8, 8, 6240, 6240, 128,
                        "f32", False, 20271),
    # short query blocks over the DiT self-attention's K/V cache (32760 tokens, 40 heads):
    # single-query decode (causal, bottom-right: the query sees every key, the last causal
    # row of xtrain's decode milestone) and 64 query rows; the split-KV forward's cases
    "dec1": Workload("dec1", "decode_sq1_over_dit_cache_h40_s32760_d128", 1, 40, 40, 1, 32760,
                     128, "bf16", True, 20269, qk_factor=0.5),
    "sq64": Workload("sq64", "sq64_over_dit_cache_h40_s32760_d128", 1, 40, 40, 64, 32760, 128,
                     "bf16", False, 20270, qk_factor=0.5),
    # profiling cases: the same kernels at sizes an ncu capture replays quickly, with
    # inputs still larger than L2 (129 MB)
    "p_self": Workload("p_self", "profile_self_s16384_h16_d128", 1, 16, 16, 16384, 16384, 128,
                       "bf16", False, 20266, qk_factor=0.5),
    "p_train": Workload("p_train", "profile_train_b8_h16_s2048_d128_causal", 8, 16, 4, 2048,
                        2048, 128, "bf16", True, 20267, has_bwd=True),
}


def get(key: str) -> Workload:
    return WORKLOADS[key]


def small_case(key: str, name: str, B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int,
               dtype: str, causal: bool, seed: int, has_bwd: bool = True,
               qk_factor: float = 1.0, lens_kind: str = "none", lens_lo: int = 0,
               lens_hi: int = 0, lens_fixed: int = 0) -> Workload:
    """A workload description for test-sized cases (same recipe, other shapes)."""
    return Workload(key, name, B, Hq, Hkv, Sq, Skv, D, dtype, causal, seed, qk_factor,
                    has_bwd, lens_kind, lens_lo, lens_hi, lens_fixed)


def make_inputs(w: Workload, with_dout: bool | None = None) -> dict:
    """Draw the workload's inputs on the CPU (contiguous tensors in the workload dtype).

    Returns a dict with ``q`` [B,Sq,Hq,D], ``k``/``v`` [B,Skv,Hkv,D], ``do`` (or None)
    and ``kv_lens`` (int32 [B, Hkv], or None when every length is Skv).
    """
    if with_dout is None:
        with_dout = w.has_bwd
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    td = w.torch_dtype

    def draw(shape, factor=1.0):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if factor != 1.0:
            x.mul_(factor)
        return x.to(td).contiguous()

    q = draw((w.B, w.Sq, w.Hq, w.D), w.qk_factor)
    k = draw((w.B, w.Skv, w.Hkv, w.D), w.qk_factor)
    v = draw((w.B, w.Skv, w.Hkv, w.D))
    do = draw((w.B, w.Sq, w.Hq, w.D)) if with_dout else None
    if w.lens_kind == "none":
        lens = None
    elif w.lens_kind == "per_head_uniform":
        lens = torch.randint(w.lens_lo, w.lens_hi + 1, (w.B, w.Hkv), generator=g,
                             dtype=torch.int64).to(torch.int32).contiguous()
    elif w.lens_kind == "fixed":
        lens = torch.full((w.B, w.Hkv), w.lens_fixed, dtype=torch.int32)
    else:  # pragma: no cover
        raise ValueError(w.lens_kind)
    return {"q": q, "k": k, "v": v, "do": do, "kv_lens": lens}


def make_paged(k, v, seq_lens, page_size: int, seed: int, spare_pages: int = 2):
    """Scatter dense K/V [B, S, Hkv, D] into shuffled page pools, as a paged cache holds them.

    Returns ``(k_pages, v_pages, block_table, max_pages)``: pools [num_pages, page_size,
    Hkv, D] in the dtype of ``k``; block_table int32 [B, max_pages] with max_pages =
    ceil(S / page_size). Only the pages that hold valid keys (t < seq_lens[b]) are
    assigned, to pages in a seeded random order; every other pool row (the tail of a
    partly filled page, unassigned and spare pages) holds NaN, and unassigned table
    entries hold -1, so that anything read past a valid length shows up.
    """
    B, S, Hkv, D = k.shape
    max_pages = -(-S // page_size)
    lens = [int(x) for x in seq_lens]
    need = [-(-L // page_size) for L in lens]
    num_pages = sum(need) + spare_pages
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    order = torch.randperm(num_pages, generator=g).tolist()
    kp = torch.full((num_pages, page_size, Hkv, D), float("nan"), dtype=k.dtype)
    vp = torch.full((num_pages, page_size, Hkv, D), float("nan"), dtype=v.dtype)
    bt = torch.full((B, max_pages), -1, dtype=torch.int32)
    used = 0
    for b in range(B):
        for t in range(need[b]):
            page = order[used]
            used += 1
            bt[b, t] = page
            n = min(page_size, lens[b] - t * page_size)
            kp[page, :n] = k[b, t * page_size:t * page_size + n]
            vp[page, :n] = v[b, t * page_size:t * page_size + n]
    return kp.contiguous(), vp.contiguous(), bt.contiguous(), max_pages
