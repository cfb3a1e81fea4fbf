"""GPU parity of the paged forward and the split-KV forward against the float64 oracle.

Paged: the K/V pools are shuffled pages whose unused rows hold NaN and whose unused
block-table entries are -1; the oracle gathers the pages itself (oracle.kvcache). Page
sizes below, at and above the kernel's 128-key tile. The paged result must also equal the
dense kernel's on the same keys bit for bit: the same tiles meet the same products.

Split-KV: single-query decode and short query blocks over long K/V, causal (bottom-right)
and not, GQA, ragged valid lengths that leave some key ranges empty, against the oracle;
the split path must really split (non-zero workspace) and be run-to-run deterministic.
"""

import numpy as np
import pytest
import torch

import oracle
from attention_sm_flash_gb300 import attn, workloads
from gpu_util import GATE, TOL, compare, run_fwd

pytestmark = pytest.mark.gpu

PAGED = [
    # key, B, Hq, Hkv, Sq, S, D, causal, page_size, valid lengths
    ("p16_d128", 3, 8, 2, 200, 700, 128, False, 16, [700, 1, 333]),
    ("p64_d64_causal_br", 2, 4, 4, 300, 300, 64, True, 64, [300, 260]),
    ("p128_gqa_causal", 2, 8, 2, 130, 1000, 128, True, 128, [1000, 517]),
    ("p256_d128", 1, 4, 1, 257, 2000, 128, False, 256, [1999]),
    ("p32_empty_seq", 2, 2, 1, 64, 96, 64, False, 32, [0, 96]),
]


@pytest.mark.parametrize("case", PAGED, ids=[c[0] for c in PAGED])
def test_paged_forward_matches_oracle_and_dense(case):
    key, B, Hq, Hkv, Sq, S, D, causal, ps, lens = case
    w = workloads.small_case(key, key, B, Hq, Hkv, Sq, S, D, "bf16", causal,
                             seed=900 + PAGED.index(case), has_bwd=False)
    inp = workloads.make_inputs(w)
    kp, vp, bt, max_pages = workloads.make_paged(inp["k"], inp["v"], lens, ps, seed=5)
    seq = torch.tensor(lens, dtype=torch.int32)
    q = inp["q"].cuda()
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, Sq), float("nan"), device="cuda")
    attn.attn_fwd_paged(q, kp.cuda(), vp.cuda(), bt.cuda(), seq.cuda(), o, lse, causal=causal,
                        scale=w.scale)
    torch.cuda.synchronize()
    assert attn.attn_peek_device_error() == (attn.ATTN_OK, 0)
    o_ref, lse_ref = oracle.kvcache.forward_paged(inp["q"], kp, vp, bt, seq, ps, w.scale, causal)
    compare(f"{key}:o", o, o_ref, *TOL["bf16"]["o"], gate=GATE["bf16"])
    compare(f"{key}:lse", lse, lse_ref, *TOL["bf16"]["lse"])
    # the dense kernel on the dense K/V with the same valid lengths
    dense_lens = torch.tensor(lens, dtype=torch.int32)[:, None].repeat(1, Hkv).contiguous()
    wd = workloads.small_case(key, key, B, Hq, Hkv, Sq, S, D, "bf16", causal, seed=0,
                              has_bwd=False)
    o_d, lse_d = run_fwd(dict(inp, kv_lens=dense_lens), wd)
    assert torch.equal(o.view(torch.int16), o_d.view(torch.int16))
    assert torch.equal(lse, lse_d)


def test_paged_bad_block_table_entry_is_flagged():
    w = workloads.small_case("pbad", "pbad", 1, 2, 2, 16, 256, 64, "bf16", False, seed=7,
                             has_bwd=False)
    inp = workloads.make_inputs(w)
    kp, vp, bt, _ = workloads.make_paged(inp["k"], inp["v"], [256], 128, seed=3)
    q, kp, vp = inp["q"].cuda(), kp.cuda(), vp.cuda()
    seq = torch.tensor([256], dtype=torch.int32).cuda()
    o, lse = torch.empty_like(q), torch.empty(1, 2, 16, device="cuda")
    bad = bt.clone()
    bad[0, 1] = kp.shape[0] + 5  # not a page of the pool
    attn.attn_fwd_paged(q, kp, vp, bad.cuda(), seq, o, lse)
    st, bits = attn.attn_peek_device_error()
    assert st == attn.ATTN_ERR_INVALID_ARG and bits & attn.ATTN_DEVERR_PAGE
    # the context stays usable: the correct table right after gives the oracle's result
    attn.attn_fwd_paged(q, kp, vp, bt.cuda(), seq, o, lse)
    torch.cuda.synchronize()
    assert attn.attn_peek_device_error() == (attn.ATTN_OK, 0)
    o_ref, lse_ref = oracle.kvcache.forward_paged(inp["q"], kp.cpu(), vp.cpu(), bt, [256], 128,
                                                  w.scale, False)
    compare("pbad:o", o, o_ref, *TOL["bf16"]["o"], gate=GATE["bf16"])


SPLIT = [
    # key, B, Hq, Hkv, Sq, Skv, D, causal, lens kind, lo, hi
    ("dec_dit_cache", 2, 40, 40, 1, 32760, 128, False, "none", 0, 0),
    ("dec_gqa_causal", 4, 8, 2, 1, 2048, 128, True, "none", 0, 0),
    ("dec3_varlen_d64", 2, 4, 2, 3, 5000, 64, True, "per_head_uniform", 0, 5000),
    ("sq64_dit_cache", 1, 40, 40, 64, 32760, 128, False, "none", 0, 0),
    ("sq128_gqa_causal", 1, 16, 4, 128, 8192, 128, True, "none", 0, 0),
]


@pytest.mark.parametrize("case", SPLIT, ids=[c[0] for c in SPLIT])
def test_splitkv_forward_matches_oracle(case):
    key, B, Hq, Hkv, Sq, Skv, D, causal, lk, lo, hi = case
    w = workloads.small_case(key, key, B, Hq, Hkv, Sq, Skv, D, "bf16", causal,
                             seed=950 + SPLIT.index(case), has_bwd=False, lens_kind=lk,
                             lens_lo=lo, lens_hi=hi)
    inp = workloads.make_inputs(w)
    need = attn.attn_fwd_splitkv_workspace_size(B, Hq, Hkv, Sq, Skv, D, attn.ATTN_BF16)
    assert need > 0  # the split path, not the dense forward
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    lens = None if inp["kv_lens"] is None else inp["kv_lens"].cuda()
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN-patterned scratch
    outs = []
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq, Sq), float("nan"), device="cuda")
        attn.attn_fwd_splitkv(q, k, v, o, lse, causal=causal, scale=w.scale, kv_lens=lens,
                              workspace=ws)
        torch.cuda.synchronize()
        assert attn.attn_peek_device_error() == (attn.ATTN_OK, 0)
        outs.append((o, lse))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1], outs[1][1])
    o_ref, lse_ref = oracle.forward(inp["q"], inp["k"], inp["v"], w.scale, causal, inp["kv_lens"])
    compare(f"{key}:o", outs[0][0], o_ref, *TOL["bf16"]["o"], gate=GATE["bf16"])
    compare(f"{key}:lse", outs[0][1], lse_ref, *TOL["bf16"]["lse"])


def test_splitkv_without_split_is_the_dense_forward():
    # enough (batch, head, query block) items: no workspace, the same call as attn_fwd
    w = workloads.small_case("nosplit", "nosplit", 2, 80, 80, 128, 1024, 64, "bf16", False,
                             seed=31, has_bwd=False)
    assert attn.attn_fwd_splitkv_workspace_size(2, 80, 80, 128, 1024, 64, attn.ATTN_BF16) == 0
    inp = workloads.make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = torch.empty_like(q), torch.empty(2, 80, 128, device="cuda")
    attn.attn_fwd_splitkv(q, k, v, o, lse, workspace=torch.empty(1, dtype=torch.uint8, device="cuda"))
    o2, lse2 = attn.forward(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16)) and torch.equal(lse, lse2)
