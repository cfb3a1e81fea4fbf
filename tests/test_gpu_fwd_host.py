"""GPU checks of the forward on pinned host tensors (attn_fwd_host): the problem goes
through the GPU in chunks of kv heads with the copies overlapped, and each chunk is an
ordinary attn_fwd on a compact sub-problem, so O and LSE must equal attn_fwd's on the same
values bit for bit (and so the oracle at the usual tolerances). Cases: GQA with per-head
valid lengths and causal masking (a last chunk with fewer heads), D = 64, fp32, more
chunks than workspace slots, a non-default stream; and the rejection of memory that is
not pinned host memory."""

import ctypes

import pytest
import torch

import oracle
from attention_sm_flash_gb300 import attn, workloads
from gpu_util import GATE, TOL, compare

pytestmark = pytest.mark.gpu

CASES = [
    # key, B, Hq, Hkv, Sq, Skv, D, dtype, causal, lens_kind (lo, hi)
    ("gqa_causal_lens", 2, 12, 6, 300, 517, 128, "bf16", True, ("per_head_uniform", 1, 517)),
    ("d64_mha", 1, 7, 7, 260, 260, 64, "bf16", False, None),
    ("f32_small", 1, 4, 2, 130, 200, 128, "f32", False, None),
    ("many_chunks", 1, 22, 11, 200, 384, 128, "bf16", True, None),
]


def _pin(t):
    return t.contiguous().pin_memory()


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_host_forward_equals_device_forward(case):
    key, B, Hq, Hkv, Sq, Skv, D, dt, causal, lk = case
    kw = {}
    if lk is not None:
        kw = dict(lens_kind=lk[0], lens_lo=lk[1], lens_hi=lk[2])
    w = workloads.small_case(key, key, B, Hq, Hkv, Sq, Skv, D, dt, causal,
                             seed=1200 + CASES.index(case), has_bwd=False, **kw)
    inp = workloads.make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    lens = None if inp["kv_lens"] is None else inp["kv_lens"].cuda()
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), device="cuda")
    attn.attn_fwd(q, k, v, o, lse, causal=causal, scale=w.scale, kv_lens=lens)

    hq, hk, hv = (_pin(inp[n]) for n in ("q", "k", "v"))
    hl = None if inp["kv_lens"] is None else _pin(inp["kv_lens"])
    ho = torch.full(inp["q"].shape, float("nan"), dtype=inp["q"].dtype).pin_memory()
    hlse = torch.full((B, Hq, Sq), float("nan")).pin_memory()
    s = torch.cuda.Stream()
    attn.attn_fwd_host(hq, hk, hv, ho, hlse, causal=causal, scale=w.scale, kv_lens=hl, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert attn.attn_peek_device_error() == (attn.ATTN_OK, 0)
    bits = torch.int16 if dt == "bf16" else torch.int32
    assert torch.equal(ho.view(bits), o.cpu().view(bits)), "O differs from attn_fwd"
    assert torch.equal(hlse.view(torch.int32), lse.cpu().view(torch.int32)), "LSE differs"
    o_ref, lse_ref = oracle.forward(inp["q"], inp["k"], inp["v"], w.scale, causal, inp["kv_lens"])
    compare(f"host_{key}:o", ho, o_ref, *TOL[dt]["o"], gate=GATE[dt])
    compare(f"host_{key}:lse", hlse, lse_ref, *TOL[dt]["lse"])


def test_host_forward_rejects_memory_that_is_not_pinned_host_memory():
    B, Hq, Hkv, Sq, Skv, D = 1, 2, 2, 64, 64, 64
    lib = attn.load()
    need = attn.attn_fwd_host_workspace_size(B, Hq, Hkv, Sq, Skv, D, attn.ATTN_BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    pinned = [torch.zeros(B, Sq, Hq, D, dtype=torch.bfloat16).pin_memory() for _ in range(4)]
    lse = torch.zeros(B, Hq, Sq).pin_memory()
    pageable = torch.zeros(B, Sq, Hq, D, dtype=torch.bfloat16)
    device = torch.zeros(B, Sq, Hq, D, dtype=torch.bfloat16, device="cuda")

    def call(q):
        return lib.attn_fwd_host(q.data_ptr(), pinned[1].data_ptr(), pinned[2].data_ptr(),
                                 pinned[3].data_ptr(), lse.data_ptr(), B, Hq, Hkv, Sq, Skv, D,
                                 0.125, 0, None, attn.ATTN_BF16, ws.data_ptr(), need, None)

    assert call(pageable) == attn.ATTN_ERR_INVALID_ARG
    assert call(device) == attn.ATTN_ERR_INVALID_ARG
    assert call(pinned[0]) == attn.ATTN_OK
    torch.cuda.synchronize()
    with pytest.raises(ValueError):
        attn.attn_fwd_host(pageable, pinned[1], pinned[2], pinned[3], lse)
