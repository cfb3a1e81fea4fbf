"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some hosts give an operator only its input and output buffers (all device memory
belongs to the host's own pool), and some latency-critical loops must not call
cudaMalloc/cudaFree because those can synchronize the device. For them the library
keeps the backward's scratch in a fixed-size array of its own. These tests call that
entry point through the C ABI and check it against the ordinary attn_bwd (which takes a
caller workspace) on two different problems in a row, so that whatever the first call
leaves in the shared array cannot leak into the second; and that a problem needing more
scratch than the array holds is refused without launching anything.

This file is collected last on purpose: it must pass both alone in a fresh process and
after every other test.
"""

import pytest
import torch

from attention_sm_flash_gb300 import attn, workloads
from gpu_util import TOL, compare

pytestmark = pytest.mark.gpu


def _inputs(key, B, Hq, Hkv, S, D, dt, causal, seed):
    w = workloads.small_case(key, key, B, Hq, Hkv, S, S, D, dt, causal, seed)
    inp = workloads.make_inputs(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    return w, dev


def test_noalloc_backward_matches_workspace_backward_two_calls_in_a_row():
    cases = [
        _inputs("na1", 2, 8, 2, 300, 128, "bf16", True, 41),
        _inputs("na2", 1, 4, 4, 520, 64, "f32", False, 42),
    ]
    for w, d in cases + cases[:1]:  # the first problem again after the second
        o, lse = attn.forward(d["q"], d["k"], d["v"], causal=w.causal, scale=w.scale)
        ref = attn.backward(d["q"], d["k"], d["v"], o, d["do"], lse, causal=w.causal,
                            scale=w.scale)
        got = [torch.full_like(t, float("nan")) for t in ref]
        attn.attn_bwd_noalloc(d["q"], d["k"], d["v"], o, d["do"], lse, *got,
                              causal=w.causal, scale=w.scale)
        torch.cuda.synchronize()
        assert attn.attn_peek_device_error() == (attn.ATTN_OK, 0)
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            compare(f"{w.key}:{name}", g, r.double().cpu().numpy(), *TOL[w.dtype]["grad"])


def test_noalloc_refuses_problems_beyond_its_scratch():
    # B * Hq * Sq rows of fp32 delta must fit in the static array; these buffers are real
    # and large enough, so nothing could be read out of bounds even if the check failed.
    rows = attn.ATTN_NOALLOC_SCRATCH_BYTES // 4 + 64
    q = torch.zeros(1, rows, 1, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 16, 1, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, rows, device="cuda")
    dq = torch.full_like(q, float("nan"))
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(k, float("nan"))
    with pytest.raises(attn.AttnError) as e:
        attn.attn_bwd_noalloc(q, k, k, q, q, lse, dq, dk, dv)
    assert e.value.status == attn.ATTN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(dk.float()).all() and torch.isnan(dq[:, :8].float()).all()
