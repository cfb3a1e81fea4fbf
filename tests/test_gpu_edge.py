"""GPU edge cases: padding that holds NaN/Inf, empty rows and sequences, determinism,
input invariance, out-of-range kv_lens, decode rows, GQA against expanded MHA,
rejected arguments and non-default streams."""

import numpy as np
import pytest
import torch

import oracle
from attention_sm_flash_gb300 import attn, workloads
from gpu_util import TOL, compare, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

DTYPES = ["bf16", "f32"]


def case(dt, B=2, Hq=4, Hkv=2, Sq=200, Skv=260, D=128, causal=False, seed=5, lens=None):
    w = workloads.small_case("e", "e", B, Hq, Hkv, Sq, Skv, D, dt, causal, seed)
    inp = workloads.make_inputs(w)
    if lens is not None:
        inp["kv_lens"] = torch.tensor(lens, dtype=torch.int32)
    return w, inp


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("causal", [False, True])
def test_padding_with_nan_and_inf_never_leaks(dt, causal):
    w, inp = case(dt, causal=causal, lens=[[260, 131], [77, 200]])
    o1, l1 = run_fwd(inp, w)
    g1 = run_bwd(inp, w, o1, l1)
    bad = dict(inp)
    k, v = inp["k"].clone(), inp["v"].clone()
    for b in range(2):
        for kvh in range(2):
            L = int(inp["kv_lens"][b, kvh])
            k[b, L:, kvh] = float("nan")
            v[b, L:, kvh] = float("inf")
    bad["k"], bad["v"] = k, v
    o2, l2 = run_fwd(bad, w)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g2 = run_bwd(bad, w, o2, l2)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
    dk, dv = g2[1].cpu(), g2[2].cpu()
    for b in range(2):
        for kvh in range(2):
            L = int(inp["kv_lens"][b, kvh])
            assert torch.all(dk[b, L:, kvh] == 0) and torch.all(dv[b, L:, kvh] == 0)


@pytest.mark.parametrize("dt", DTYPES)
def test_empty_rows_and_sequences(dt):
    # causal, bottom-right: with L < Sq the first Sq - L rows see nothing; L = 0 is empty
    w, inp = case(dt, B=1, Hq=4, Hkv=2, Sq=300, Skv=300, D=64, causal=True, lens=[[0, 170]])
    o, lse = run_fwd(inp, w)
    o_ref, lse_ref = oracle.forward(inp["q"], inp["k"], inp["v"], w.scale, True, inp["kv_lens"])
    compare("o", o, o_ref, *TOL[dt]["o"])
    compare("lse", lse, lse_ref, *TOL[dt]["lse"])
    oc, lc = o.cpu(), lse.cpu()
    assert torch.all(oc[0, :, 0:2] == 0) and torch.all(torch.isneginf(lc[0, 0:2]))
    assert torch.all(oc[0, :130, 2:4] == 0) and torch.all(torch.isneginf(lc[0, 2:4, :130]))
    dq, dk, dv = run_bwd(inp, w, o, lse)
    ref = oracle.backward(inp["q"], inp["k"], inp["v"], inp["do"], w.scale, True, inp["kv_lens"])
    for n, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref[:3]):
        compare(n, got, r, *TOL[dt]["grad"])
    assert torch.all(dq.cpu()[0, :, 0:2] == 0)


@pytest.mark.parametrize("dt", DTYPES)
def test_no_keys_at_all(dt):
    w, inp = case(dt, B=1, Hq=2, Hkv=2, Sq=70, Skv=0, D=64)
    o, lse = run_fwd(inp, w)
    assert torch.all(o.cpu() == 0) and torch.all(torch.isneginf(lse.cpu()))
    dq, dk, dv = run_bwd(inp, w, o, lse)
    assert torch.all(dq.cpu() == 0)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("causal", [False, True])
def test_bitwise_deterministic_and_inputs_unchanged(dt, causal):
    w, inp = case(dt, B=1, Hq=8, Hkv=2, Sq=520, Skv=520, D=128, causal=causal)
    keep = {k: (v.clone() if v is not None else None) for k, v in inp.items()}
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    outs = []
    for _ in range(2):
        o, lse = attn.forward(dev["q"], dev["k"], dev["v"], causal=causal, scale=w.scale)
        dq, dk, dv = attn.backward(dev["q"], dev["k"], dev["v"], o, dev["do"], lse,
                                   causal=causal, scale=w.scale)
        outs.append([t.clone() for t in (o, lse, dq, dk, dv)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    for k in ("q", "k", "v", "do"):
        assert torch.equal(dev[k].cpu(), keep[k])


@pytest.mark.parametrize("dt", DTYPES)
def test_out_of_range_kv_lens_are_clamped_and_flagged(dt):
    w, inp = case(dt, B=1, Hq=2, Hkv=2, Sq=64, Skv=100, D=64, lens=[[130, -4]])
    q, k, v = inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda()
    attn.attn_peek_device_error()  # start from a clear word
    o, lse = attn.forward(q, k, v, scale=w.scale, kv_lens=inp["kv_lens"].cuda())
    st, bits = attn.attn_peek_device_error()
    assert st == attn.ATTN_ERR_INVALID_ARG and bits & attn.ATTN_DEVERR_KVLEN
    o2, l2 = attn.forward(q, k, v, scale=w.scale,
                          kv_lens=torch.tensor([[100, 0]], dtype=torch.int32, device="cuda"))
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    assert attn.attn_peek_device_error() == (attn.ATTN_OK, 0)


@pytest.mark.parametrize("dt", DTYPES)
def test_decode_rows_match_last_causal_rows(dt):
    w, inp = case(dt, B=1, Hq=4, Hkv=1, Sq=333, Skv=333, D=128, causal=True)
    o_full, l_full = run_fwd(inp, w)
    dec = dict(inp)
    dec["q"] = inp["q"][:, -3:].contiguous()
    wd = workloads.small_case("d", "d", 1, 4, 1, 3, 333, 128, dt, True, 0)
    o_dec, l_dec = run_fwd(dec, wd)
    tol = TOL[dt]
    compare("o_dec", o_dec, o_full[:, -3:].double().cpu().numpy(), *tol["o"])
    compare("lse_dec", l_dec, l_full[:, :, -3:].double().cpu().numpy(), *tol["lse"])


@pytest.mark.parametrize("dt", DTYPES)
def test_gqa_matches_mha_on_expanded_kv(dt):
    w, inp = case(dt, B=2, Hq=8, Hkv=2, Sq=150, Skv=150, D=64, causal=True)
    o, lse = run_fwd(inp, w)
    dq, dk, dv = run_bwd(inp, w, o, lse)
    ex = dict(inp)
    ex["k"] = inp["k"].repeat_interleave(4, dim=2).contiguous()
    ex["v"] = inp["v"].repeat_interleave(4, dim=2).contiguous()
    we = workloads.small_case("x", "x", 2, 8, 8, 150, 150, 64, dt, True, 0)
    o2, l2 = run_fwd(ex, we)
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    dq2, dk2, dv2 = run_bwd(ex, we, o2, l2)
    assert torch.equal(dq, dq2)
    tol = TOL[dt]["grad"]
    sum_k = dk2.double().cpu().view(2, 150, 2, 4, 64).sum(3).numpy()
    sum_v = dv2.double().cpu().view(2, 150, 2, 4, 64).sum(3).numpy()
    compare("dk_group_sum", dk, sum_k, *tol)
    compare("dv_group_sum", dv, sum_v, *tol)


def test_rejected_arguments_launch_nothing():
    q = torch.randn(1, 64, 2, 64, device="cuda").to(torch.bfloat16)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((1, 2, 64), float("nan"), device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd(q, q[:, :, :1].contiguous(), q[:, :, :1].contiguous(), o, lse,
                      scale=float("nan"))
    assert e.value.status == attn.ATTN_ERR_INVALID_ARG
    qq = torch.randn(1, 64, 2, 96, device="cuda").to(torch.bfloat16)
    with pytest.raises(attn.AttnError) as e:
        attn.forward(qq, qq, qq)
    assert e.value.status == attn.ATTN_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.isnan(o.float()).all() and torch.isnan(lse).all()


@pytest.mark.parametrize("dt", DTYPES)
def test_non_default_stream(dt):
    w, inp = case(dt, B=1, Hq=2, Hkv=2, Sq=256, Skv=256, D=128, causal=True)
    s = torch.cuda.Stream()
    q, k, v = inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        o, lse = attn.forward(q, k, v, causal=True, scale=w.scale, stream=s)
    s.synchronize()
    o_ref, lse_ref = oracle.forward(inp["q"], inp["k"], inp["v"], w.scale, True)
    compare("o", o, o_ref, *TOL[dt]["o"])
    compare("lse", lse, lse_ref, *TOL[dt]["lse"])


def test_bounded_wait_runs_out_reports_timeout_and_gpu_stays_usable():
    """A forward whose producer skips one load (test-only injection): the consumer's
    bounded wait runs out, the kernel records a timeout and returns, and the next call
    on the same context is correct."""
    w, inp = case("bf16", B=1, Hq=2, Hkv=2, Sq=256, Skv=256, D=128)
    q, k, v = inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda()
    torch.cuda.synchronize()
    attn.attn_peek_device_error()
    attn.attn_test_inject_fault(1, 200)
    attn.forward(q, k, v, scale=w.scale)
    st, bits = attn.attn_peek_device_error()
    assert st == attn.ATTN_ERR_TIMEOUT and bits & attn.ATTN_DEVERR_TIMEOUT
    o, lse = run_fwd(inp, w)
    o_ref, lse_ref = oracle.forward(inp["q"], inp["k"], inp["v"], w.scale, False)
    compare("o_after_timeout", o, o_ref, *TOL["bf16"]["o"])
    compare("lse_after_timeout", lse, lse_ref, *TOL["bf16"]["lse"])


@pytest.mark.parametrize("D", [64, 128])
def test_gradients_at_16_byte_aligned_outputs(D):
    """dQ, dK, dV at addresses 16-byte but not 32-byte aligned (the API's minimum) get the
    same bits as at aligned ones (the kernels fall back from 32-byte to 16-byte stores)."""
    w, inp = case("bf16", B=1, Hq=4, Hkv=4, Sq=300, Skv=300, D=D, causal=True)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    o, lse = attn.forward(dev["q"], dev["k"], dev["v"], causal=True, scale=w.scale)
    ref = attn.backward(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, causal=True,
                        scale=w.scale)
    outs = []
    for t in (dev["q"], dev["k"], dev["v"]):
        buf = torch.empty(t.numel() + 8, dtype=t.dtype, device="cuda")
        view = buf[8:8 + t.numel()].view(t.shape)
        assert view.data_ptr() % 32 == 16
        outs.append(view)
    attn.attn_bwd(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, *outs, causal=True,
                  scale=w.scale, kv_lens=None)
    torch.cuda.synchronize()
    st, bits = attn.attn_peek_device_error()
    assert st == attn.ATTN_OK, (st, bits)
    for name, a, b in zip(("dq", "dk", "dv"), outs, ref):
        assert torch.equal(a, b), name
