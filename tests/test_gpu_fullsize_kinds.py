"""Parity of the split-KV and paged forwards at the full sizes that bench.py times, in the
same launch configuration (the same entry points on the same workloads):

* decode over the DiT cache (one query row per head, 32760 keys, 40 heads, causal) through
  the split-KV forward, against the whole oracle;
* 64 query rows over the same cache through the split-KV forward, against the whole oracle;
* the DiT self-attention through a 256-key paged cache with a shuffled block table: equal
  bit for bit to the dense forward on the same keys, and the oracle on sampled rows;
* the DiT self-attention from pinned host tensors (attn_fwd_host, the e2e call): equal bit
  for bit to the dense forward.

The scores are small (Q and K scaled by 0.5, so the softmax over 32760 keys is nearly
uniform and |O| is about 0.005); the rel-L2 and max|diff|/max|ref| gates keep the checks
from passing on a near-zero O.
"""

import numpy as np
import pytest
import torch

import oracle
from attention_sm_flash_gb300 import attn, workloads
from gpu_util import GATE, TOL, compare

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("key", ["dec1", "sq64"])
def test_split_kv_full_size_against_the_whole_oracle(key):
    w = workloads.get(key)
    inp = workloads.make_inputs(w)
    need = attn.attn_fwd_splitkv_workspace_size(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, attn.ATTN_BF16)
    assert need > 0  # the split path, as bench.py times it
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.Hq, w.Sq), float("nan"), device="cuda")
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    attn.attn_fwd_splitkv(q, k, v, o, lse, causal=w.causal, scale=w.scale, workspace=ws)
    torch.cuda.synchronize()
    assert attn.attn_peek_device_error() == (attn.ATTN_OK, 0)
    o_ref, lse_ref = oracle.forward(inp["q"], inp["k"], inp["v"], w.scale, w.causal, None)
    compare(f"{key}:o", o.cpu(), o_ref, *TOL["bf16"]["o"], gate=GATE["bf16"])
    compare(f"{key}:lse", lse.cpu(), lse_ref, *TOL["bf16"]["lse"])


def test_paged_dit_self_attention_full_size():
    w = workloads.get("c4")
    inp = workloads.make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Sq), device="cuda")
    attn.attn_fwd(q, k, v, o, lse, causal=w.causal, scale=w.scale)
    del k, v
    kp, vp, bt, _ = workloads.make_paged(inp["k"], inp["v"], [w.Skv] * w.B, 256, seed=w.seed)
    kp, vp, bt = kp.cuda(), vp.cuda(), bt.cuda()
    seq = torch.full((w.B,), w.Skv, dtype=torch.int32, device="cuda")
    op = torch.full_like(q, float("nan"))
    lsep = torch.full((w.B, w.Hq, w.Sq), float("nan"), device="cuda")
    attn.attn_fwd_paged(q, kp, vp, bt, seq, op, lsep, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert attn.attn_peek_device_error() == (attn.ATTN_OK, 0)
    assert torch.equal(op.view(torch.int16), o.view(torch.int16)), "paged O differs from dense"
    assert torch.equal(lsep.view(torch.int32), lse.view(torch.int32)), "paged LSE differs"
    op, lsep = op.cpu(), lsep.cpu()
    r = np.random.default_rng(7)
    for h in (0, 13, 27, 39):
        rows = np.unique(np.concatenate([[0, 127, 128, w.Sq - 1], r.choice(w.Sq, 28, replace=False)]))
        o_ref, lse_ref = oracle.forward_rows(inp["q"][:, :, h:h + 1], inp["k"][:, :, h:h + 1],
                                             inp["v"][:, :, h:h + 1], w.scale, w.causal, None,
                                             0, 0, rows)
        compare(f"c4_paged256:o[h={h}]", op[0, rows, h], o_ref, *TOL["bf16"]["o"], gate=GATE["bf16"])
        compare(f"c4_paged256:lse[h={h}]", lsep[0, h, rows], lse_ref, *TOL["bf16"]["lse"])


def test_host_forward_dit_self_attention_full_size():
    """The call bench.py times for the e2e figure of the DiT self-attention: attn_fwd_host
    on pinned host tensors (five chunks of eight heads, copies overlapped with the compute)
    gives attn_fwd's O and LSE bit for bit."""
    w = workloads.get("c4")
    inp = workloads.make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Sq), device="cuda")
    attn.attn_fwd(q, k, v, o, lse, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    o, lse = o.cpu(), lse.cpu()
    del q, k, v
    hq, hk, hv = (inp[n].pin_memory() for n in ("q", "k", "v"))
    ho = torch.full(inp["q"].shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    hlse = torch.full((w.B, w.Hq, w.Sq), float("nan")).pin_memory()
    attn.attn_fwd_host(hq, hk, hv, ho, hlse, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert attn.attn_peek_device_error() == (attn.ATTN_OK, 0)
    assert torch.equal(ho.view(torch.int16), o.view(torch.int16)), "host-path O differs"
    assert torch.equal(hlse.view(torch.int32), lse.view(torch.int32)), "host-path LSE differs"
