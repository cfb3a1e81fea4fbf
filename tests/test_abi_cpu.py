"""The C-ABI library loads and exports every symbol include/attn.h declares, and its
host-side argument checks reject bad calls before touching CUDA (no GPU needed)."""

import ctypes
import os
import re

import pytest

from attention_sm_flash_gb300 import attn
from attention_sm_flash_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return attn.load()


def declared_functions():
    with open(os.path.join(ROOT, "include", "attn.h")) as f:
        text = f.read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(attn.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_build_info(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert attn.status_string(code).startswith("ATTN_")
    assert "sm_103a" in attn.build_info()


def test_workspace_size(lib):
    # MHA: delta only
    n = attn.attn_bwd_workspace_size(8, 12, 12, 1024, 1024, 64, attn.ATTN_BF16)
    assert n == 8 * 12 * 1024 * 4
    # GQA with few (batch, kv head, key tile) items: delta + fp32 partial dK, dV of P
    # parts per group. 4 x 2 x 16 = 128 items: P = 2 (the smallest divisor of the group
    # size 4 giving >= 256 items)
    n = attn.attn_bwd_workspace_size(4, 8, 2, 2048, 2048, 128, attn.ATTN_BF16)
    assert n == 4 * 8 * 2048 * 4 + 2 * 4 * 2048 * (2 * 2) * 128 * 4 and n % 256 == 0
    # 1 x 1 x 3 items, group of 4: no divisor reaches 256, one part per query head
    n = attn.attn_bwd_workspace_size(1, 4, 1, 257, 257, 128, attn.ATTN_BF16)
    assert n == 256 * (-(-(4 * 257 * 4) // 256)) + 2 * 256 * (-(-(257 * 4 * 128 * 4) // 256))
    # 1 x 1 x 65 items, group of 8: P = 4 (65 x 2 < 256 <= 65 x 4)
    n = attn.attn_bwd_workspace_size(1, 8, 1, 130, 8200, 64, attn.ATTN_BF16)
    assert n == 256 * (-(-(8 * 130 * 4) // 256)) + 2 * 256 * (-(-(8200 * 4 * 64 * 4) // 256))
    # many items, or fp32: delta only
    assert attn.attn_bwd_workspace_size(64, 8, 2, 2048, 2048, 128, attn.ATTN_BF16) == 64 * 8 * 2048 * 4
    assert attn.attn_bwd_workspace_size(4, 8, 2, 2048, 2048, 128, attn.ATTN_F32) == 4 * 8 * 2048 * 4
    assert attn.attn_bwd_workspace_size(0, 8, 2, 2048, 2048, 128, attn.ATTN_BF16) == 0


A = 0x10000  # a fake, 256-byte aligned "device address": never dereferenced here


def fwd(lib, **kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, Hq=2, Hkv=2, Sq=8, Skv=8, D=64, scale=0.125,
                causal=0, kv_lens=None, dtype=attn.ATTN_BF16, stream=None)
    args.update(kw)
    return lib.attn_fwd(*args.values())


def bwd(lib, **kw):
    args = dict(q=A, k=A, v=A, o=A, do=A, lse=A, dq=A, dk=A, dv=A, B=1, Hq=2, Hkv=2, Sq=8,
                Skv=8, D=64, scale=0.125, causal=0, kv_lens=None, dtype=attn.ATTN_BF16,
                ws=A, ws_bytes=1 << 20, stream=None)
    args.update(kw)
    return lib.attn_bwd(*args.values())


@pytest.mark.parametrize("kw,want", [
    (dict(Hq=3, Hkv=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(Hkv=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(Sq=-5), attn.ATTN_ERR_INVALID_ARG),
    (dict(Skv=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(D=256), attn.ATTN_ERR_UNSUPPORTED),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), attn.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(dtype=7), attn.ATTN_ERR_INVALID_ARG),
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(o=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(lse=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(q=A + 8), attn.ATTN_ERR_INVALID_ARG),
    (dict(k=A + 2), attn.ATTN_ERR_INVALID_ARG),
    (dict(lse=A + 2), attn.ATTN_ERR_INVALID_ARG),
    (dict(kv_lens=A + 1), attn.ATTN_ERR_INVALID_ARG),
    (dict(Hq=70000, Hkv=1), attn.ATTN_ERR_UNSUPPORTED),
])
def test_fwd_rejects_bad_arguments(lib, kw, want):
    assert fwd(lib, **kw) == want


def test_empty_problems_are_a_no_op(lib):
    assert fwd(lib, B=0) == attn.ATTN_OK
    assert fwd(lib, Sq=0, q=None, o=None, lse=None) == attn.ATTN_OK
    assert bwd(lib, B=0) == attn.ATTN_OK
    assert bwd(lib, Sq=0, Skv=0) == attn.ATTN_OK


@pytest.mark.parametrize("kw,want", [
    (dict(ws=None), attn.ATTN_ERR_WORKSPACE),
    (dict(ws_bytes=100), attn.ATTN_ERR_WORKSPACE),
    (dict(ws=A + 16), attn.ATTN_ERR_WORKSPACE),
    (dict(dq=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(do=A + 4), attn.ATTN_ERR_INVALID_ARG),
    (dict(dv=A + 4), attn.ATTN_ERR_INVALID_ARG),
    (dict(Hq=4, Hkv=3), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=32), attn.ATTN_ERR_UNSUPPORTED),
])
def test_bwd_rejects_bad_arguments(lib, kw, want):
    assert bwd(lib, **kw) == want


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q, q, q.clone(), torch.zeros(1, 2, 8))


def test_noalloc_rejects_oversize_before_touching_cuda(lib):
    rows = attn.ATTN_NOALLOC_SCRATCH_BYTES // 4 + 64
    st = lib.attn_bwd_noalloc(A, A, A, A, A, A, A, A, A, 1, 1, 1, rows, 16, 64, 0.125, 0,
                              None, attn.ATTN_BF16, None)
    assert st == attn.ATTN_ERR_WORKSPACE


def test_noalloc_limit_counts_the_split_gqa_partials(lib):
    # the GQA training shape has only 65,536 query rows (256 KiB of delta), but its split
    # group adds two fp32 partial buffers: about 33.8 MB in all, beyond the 8 MiB array
    need = attn.attn_bwd_workspace_size(4, 8, 2, 2048, 2048, 128, attn.ATTN_BF16)
    assert need > attn.ATTN_NOALLOC_SCRATCH_BYTES > 4 * 8 * 2048 * 4
    st = lib.attn_bwd_noalloc(A, A, A, A, A, A, A, A, A, 4, 8, 2, 2048, 2048, 128, 0.088, 1,
                              None, attn.ATTN_BF16, None)
    assert st == attn.ATTN_ERR_WORKSPACE


def _meta(shape, dtype):
    """A tensor that passes the binding's device check without a GPU (the shape and
    dtype checks run before anything reaches the library)."""
    import torch

    class FakeDev(torch.Tensor):
        pass

    t = torch.zeros(shape, dtype=dtype)
    t.__class__ = FakeDev
    FakeDev.is_cuda = property(lambda self: True)
    return t


@pytest.mark.parametrize("bad", ["lse_dtype", "lse_shape", "lens_dtype", "lens_shape",
                                 "o_shape", "k_dtype", "v_shape", "kd_mismatch"])
def test_binding_checks_shapes_and_dtypes_fwd(bad):
    import torch
    bf = torch.bfloat16
    q, k, v = _meta((2, 16, 4, 64), bf), _meta((2, 24, 2, 64), bf), _meta((2, 24, 2, 64), bf)
    o, lse = _meta((2, 16, 4, 64), bf), _meta((2, 4, 16), torch.float32)
    lens = _meta((2, 2), torch.int32)
    if bad == "lse_dtype":
        lse = _meta((2, 4, 16), bf)
    elif bad == "lse_shape":
        lse = _meta((2, 16, 4), torch.float32)
    elif bad == "lens_dtype":
        lens = _meta((2, 2), torch.int64)
    elif bad == "lens_shape":
        lens = _meta((2,), torch.int32)
    elif bad == "o_shape":
        o = _meta((2, 16, 2, 64), bf)
    elif bad == "k_dtype":
        k = _meta((2, 24, 2, 64), torch.float32)
    elif bad == "v_shape":
        v = _meta((2, 23, 2, 64), bf)
    elif bad == "kd_mismatch":
        k, v = _meta((2, 24, 2, 128), bf), _meta((2, 24, 2, 128), bf)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, k, v, o, lse, kv_lens=lens)


@pytest.mark.parametrize("bad", ["dq", "dk", "dv", "dout"])
def test_binding_checks_shapes_and_dtypes_bwd(bad):
    import torch
    bf = torch.bfloat16
    t = {n: _meta((1, 16, 4, 64), bf) for n in ("q", "o", "dout", "dq")}
    t.update({n: _meta((1, 24, 2, 64), bf) for n in ("k", "v", "dk", "dv")})
    lse = _meta((1, 4, 16), torch.float32)
    t[bad] = _meta(t[bad].shape, torch.float32)
    with pytest.raises(ValueError):
        attn.attn_bwd(t["q"], t["k"], t["v"], t["o"], t["dout"], lse, t["dq"], t["dk"], t["dv"])
    with pytest.raises(ValueError):
        attn.attn_bwd_noalloc(t["q"], t["k"], t["v"], t["o"], t["dout"], lse, t["dq"], t["dk"],
                              t["dv"])


def paged(lib, **kw):
    args = dict(q=A, kp=A, vp=A, bt=A, lens=A, o=A, lse=A, B=2, Hq=4, Hkv=2, Sq=8, pages=6,
                page_size=128, max_pages=3, D=128, scale=0.088, causal=0,
                dtype=attn.ATTN_BF16, stream=None)
    args.update(kw)
    return lib.attn_fwd_paged(*args.values())


@pytest.mark.parametrize("kw,want", [
    (dict(page_size=48), attn.ATTN_ERR_UNSUPPORTED),
    (dict(page_size=8), attn.ATTN_ERR_UNSUPPORTED),
    (dict(page_size=200), attn.ATTN_ERR_UNSUPPORTED),
    (dict(page_size=384), attn.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=attn.ATTN_F32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(D=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(pages=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(max_pages=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(page_size=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(max_pages=1 << 24, page_size=1 << 10), attn.ATTN_ERR_INVALID_ARG),
    (dict(bt=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(kp=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(bt=A + 2), attn.ATTN_ERR_INVALID_ARG),
    (dict(lens=A + 1), attn.ATTN_ERR_INVALID_ARG),
    (dict(vp=A + 8), attn.ATTN_ERR_INVALID_ARG),
    (dict(Hq=3), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
])
def test_paged_rejects_bad_arguments(lib, kw, want):
    assert paged(lib, **kw) == want


def test_paged_empty_problem_is_a_no_op(lib):
    assert paged(lib, B=0) == attn.ATTN_OK
    assert paged(lib, Sq=0, q=None, o=None) == attn.ATTN_OK


def test_splitkv_workspace_size(lib):
    f = attn.attn_fwd_splitkv_workspace_size

    def r256(n):
        return (n + 255) // 256 * 256
    # decode over the DiT cache: 40 (batch, head) items -> 7 ranges of 37 key tiles
    # (280 items: 2 nearly full rounds on 152 SMs; 8 ranges would give 320, 2.1 rounds)
    assert f(1, 40, 40, 1, 32760, 128, attn.ATTN_BF16) == r256(7 * 40 * 128 * 4) + r256(7 * 40 * 4)
    # 64 query rows: still one query block per head
    assert f(1, 40, 40, 64, 32760, 128, attn.ATTN_BF16) == r256(7 * 40 * 64 * 128 * 4) + r256(7 * 40 * 64 * 4)
    # 16 items over 4096 keys: 8 ranges of 4 tiles (128 items, one round)
    assert f(1, 16, 16, 1, 4096, 128, attn.ATTN_BF16) == r256(8 * 16 * 128 * 4) + r256(8 * 16 * 4)
    # one head, short K/V: at least 4 tiles per range (9 tiles -> 2 ranges)
    assert f(1, 1, 1, 1, 9 * 128, 64, attn.ATTN_BF16) == 2 * 64 * 4 + 256
    # enough items without splitting, fp32, tiny K/V, empty problems: no workspace
    assert f(1, 40, 40, 32760, 32760, 128, attn.ATTN_BF16) == 0
    assert f(1, 40, 40, 1, 32760, 128, attn.ATTN_F32) == 0
    assert f(1, 1, 1, 1, 300, 128, attn.ATTN_BF16) == 0
    assert f(0, 40, 40, 1, 32760, 128, attn.ATTN_BF16) == 0


def test_splitkv_needs_its_workspace(lib):
    def call(**kw):
        args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, Hq=40, Hkv=40, Sq=1, Skv=32760, D=128,
                    scale=0.088, causal=0, lens=None, dtype=attn.ATTN_BF16, ws=A,
                    ws_bytes=1 << 20, stream=None)
        args.update(kw)
        return lib.attn_fwd_splitkv(*args.values())
    assert call(ws=None) == attn.ATTN_ERR_WORKSPACE
    assert call(ws_bytes=1000) == attn.ATTN_ERR_WORKSPACE
    assert call(ws=A + 64) == attn.ATTN_ERR_WORKSPACE
    assert call(D=80) == attn.ATTN_ERR_UNSUPPORTED
    assert call(q=A + 4) == attn.ATTN_ERR_INVALID_ARG
    assert call(B=0) == attn.ATTN_OK


def test_fwd_host_workspace_size(lib):
    f = attn.attn_fwd_host_workspace_size

    def r256(n):
        return (n + 255) // 256 * 256

    # the DiT self-attention: 40 kv heads in 5 chunks of 8; two slots, each one chunk's
    # Q, K, V, O (bf16), LSE and valid lengths
    B, H, S, D = 1, 40, 32760, 128
    slot = 4 * r256(B * S * 8 * D * 2) + r256(B * 8 * S * 4) + r256(B * 8 * 4)
    assert f(B, H, H, S, S, D, attn.ATTN_BF16) == 2 * slot
    # GQA 8 query heads on 2 kv heads: chunks of one kv head with its 4 query heads, fp32
    B, Sq, Skv = 2, 100, 300
    slot = (2 * r256(B * Sq * 4 * 64 * 4) + 2 * r256(B * Skv * 1 * 64 * 4) +
            r256(B * 4 * Sq * 4) + r256(B * 1 * 4))
    assert f(B, 8, 2, Sq, Skv, 64, attn.ATTN_F32) == 2 * slot
    # empty problems and unsupported sizes need none
    assert f(0, 40, 40, 10, 10, 128, attn.ATTN_BF16) == 0
    assert f(1, 40, 40, 0, 10, 128, attn.ATTN_BF16) == 0
    assert f(1, 40, 40, 10, 10, 80, attn.ATTN_BF16) == 0
    assert f(1, 6, 4, 10, 10, 128, attn.ATTN_BF16) == 0


def test_fwd_host_argument_checks(lib):
    def call(**kw):
        args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, Hq=40, Hkv=40, Sq=64, Skv=64, D=128,
                    scale=0.088, causal=0, lens=None, dtype=attn.ATTN_BF16, ws=A,
                    ws_bytes=1 << 40, stream=None)
        args.update(kw)
        return lib.attn_fwd_host(*args.values())
    assert call(Hq=6, Hkv=4) == attn.ATTN_ERR_INVALID_ARG
    assert call(D=80) == attn.ATTN_ERR_UNSUPPORTED
    assert call(scale=float("nan")) == attn.ATTN_ERR_INVALID_ARG
    assert call(causal=2) == attn.ATTN_ERR_INVALID_ARG
    assert call(q=None) == attn.ATTN_ERR_INVALID_ARG
    assert call(ws=None) == attn.ATTN_ERR_WORKSPACE
    assert call(ws_bytes=4096) == attn.ATTN_ERR_WORKSPACE
    assert call(ws=A + 64) == attn.ATTN_ERR_WORKSPACE
    assert call(B=0) == attn.ATTN_OK
    assert call(Sq=0) == attn.ATTN_OK


def test_source_digest_covers_code_not_comments():
    """The key of the recorded DRAM-traffic figures changes with the code only: comments and
    layout are dropped, string and character literals are kept whole."""
    from attention_sm_flash_gb300.build import _code_text
    a = b'int a = 1; // a "note"\n/* block\n   comment */ const char* s = "x // y /* z */";\n'
    b = b'int  a = 1;\n\n const char* s = "x // y /* z */"; // other note\n'
    assert _code_text(a) == _code_text(b) == b'int a = 1; const char* s = "x // y /* z */";'
    assert _code_text(b"char q = '\"'; int b; // c") == b"char q = '\"'; int b;"
    assert _code_text(b"int a = 1;") != _code_text(b"int a = 2;")
    assert _code_text(b'puts("a\\" // b");') == b'puts("a\\" // b");'


def test_backward_per_kernel_estimates_follow_the_recorded_shares(monkeypatch):
    """bench.py's per-kernel backward figures: the recorded ncu shares scaled to the call's
    time, GEMM FLOPs over each kernel's share; none once the backward's code changes."""
    import bench
    from attention_sm_flash_gb300 import build as libbuild
    fwd_fl = 3.4376e10
    est = bench.bwd_kernel_estimates("c3", "bf16", 0.14, fwd_fl, 1944.9)
    assert est is not None and [e["kernel"].split("<")[0] for e in est] == [
        "bwd_delta_kernel", "bwd_dq_sm103_kernel", "bwd_dkdv_sm103_kernel", "bwd_group_reduce_kernel"]
    assert abs(sum(e["ncu_share"] for e in est) - 1.0) < 1e-3
    assert abs(sum(e["ms_est"] for e in est) - 0.14) < 1e-4
    dkdv = est[2]
    assert dkdv["gemms"] == 4
    want = 4 * fwd_fl / 2 / (dkdv["ms_est"] * 1e-3) / 1e12
    assert abs(dkdv["tflops_est"] - want) < 0.1 and abs(dkdv["frac_est"] - want / 1944.9) < 1e-4
    assert est[0]["tflops_est"] is None  # no GEMM in the delta kernel
    assert bench.bwd_kernel_estimates("c1", "f32", 0.1, 1e6, 1.0) is None  # no record
    monkeypatch.setattr(libbuild, "source_digest", lambda *a, **k: "0000000000000000")
    assert bench.bwd_kernel_estimates("c3", "bf16", 0.14, fwd_fl, 1944.9) is None
