"""Thin ctypes binding of libattn (include/attn.h), with the C ABI's names.

Argument marshalling only: tensors become device pointers and sizes, the stream
becomes a handle, a negative status becomes an exception. Every step of the
computation runs in the library's CUDA kernels; there is no CPU path and no fallback.
If the library has not been built the first call raises.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libattn.so")

ATTN_BF16 = 0
ATTN_F32 = 1
ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_CUDA = -3
ATTN_ERR_TIMEOUT = -4
ATTN_ERR_WORKSPACE = -5
ATTN_DEVERR_KVLEN = 0x1
ATTN_DEVERR_TIMEOUT = 0x2
ATTN_DEVERR_LAYOUT = 0x4
ATTN_DEVERR_PAGE = 0x8

EXPORTED = ("attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_peek_device_error",
            "attn_status_string", "attn_build_info", "attn_launch_count", "attn_bwd_noalloc",
            "attn_test_inject_fault", "attn_last_cuda_error", "attn_fwd_paged",
            "attn_fwd_splitkv", "attn_fwd_splitkv_workspace_size", "attn_fwd_host",
            "attn_fwd_host_workspace_size")
ATTN_NOALLOC_SCRATCH_BYTES = 8 << 20

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        extra = ""
        if status == ATTN_ERR_CUDA:
            extra = ": " + load().attn_last_cuda_error().decode()
        super().__init__(f"{what}: {status_string(status)} ({status}){extra}")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libattn.so (once) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libattn.so is not built ({path}); run "
                           "`python -m attention_sm_flash_gb300.build` first")
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_fwd.restype = i
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, i, vp]
    lib.attn_bwd.restype = i
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp,
                             i, vp, sz, vp]
    lib.attn_bwd_workspace_size.restype = sz
    lib.attn_bwd_workspace_size.argtypes = [i, i, i, i, i, i, i]
    lib.attn_peek_device_error.restype = i
    lib.attn_peek_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_status_string.argtypes = [i]
    lib.attn_build_info.restype = ctypes.c_char_p
    lib.attn_build_info.argtypes = []
    lib.attn_last_cuda_error.restype = ctypes.c_char_p
    lib.attn_last_cuda_error.argtypes = []
    lib.attn_launch_count.restype = ctypes.c_uint64
    lib.attn_test_inject_fault.restype = None
    lib.attn_test_inject_fault.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
    lib.attn_bwd_noalloc.restype = i
    lib.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i,
                                     vp, i, vp]
    lib.attn_launch_count.argtypes = []
    lib.attn_fwd_paged.restype = i
    lib.attn_fwd_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, i,
                                   vp]
    lib.attn_fwd_splitkv.restype = i
    lib.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, i, vp, sz,
                                     vp]
    lib.attn_fwd_splitkv_workspace_size.restype = sz
    lib.attn_fwd_splitkv_workspace_size.argtypes = [i, i, i, i, i, i, i]
    lib.attn_fwd_host.restype = i
    lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, i, vp, sz, vp]
    lib.attn_fwd_host_workspace_size.restype = sz
    lib.attn_fwd_host_workspace_size.argtypes = [i, i, i, i, i, i, i]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def build_info() -> str:
    return load().attn_build_info().decode()


def attn_launch_count() -> int:
    """Kernel launches the library has issued in this process."""
    return int(load().attn_launch_count())


def attn_test_inject_fault(mask: int, timeout_ms: int = 0) -> None:
    """Test-only: the next bf16 forward launch injects a fault (see include/attn.h)."""
    load().attn_test_inject_fault(int(mask), int(timeout_ms))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float32:
        return ATTN_F32
    raise TypeError(f"unsupported element type {t.dtype}")


def _check_cuda(*ts):
    for t in ts:
        if t is not None and not isinstance(t, int):
            if not t.is_cuda:
                raise ValueError("libattn takes device tensors only")
            if not t.is_contiguous():
                raise ValueError("libattn takes contiguous tensors only")


def _check_shapes(q, k, v, lse, kv_lens, like_q=(), like_k=()):
    """Shapes and element types the C ABI assumes but cannot see through raw pointers:
    q [B,Sq,Hq,D]; k, v [B,Skv,Hkv,D]; every data tensor one element type; lse fp32
    [B,Hq,Sq]; kv_lens int32 [B,Hkv]. ``like_q`` / ``like_k``: (name, tensor) pairs that
    must have q's / k's shape and element type."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, S, H, D]")
    B, Sq, Hq, D = q.shape
    if k.shape[0] != B or k.shape[3] != D:
        raise ValueError(f"k {tuple(k.shape)} does not match q {tuple(q.shape)} in B or D")
    if v.shape != k.shape:
        raise ValueError(f"v {tuple(v.shape)} differs from k {tuple(k.shape)}")
    for name, t in (("k", k), ("v", v)):
        if t.dtype != q.dtype:
            raise ValueError(f"{name} is {t.dtype}, q is {q.dtype}")
    for name, t in like_q:
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must be {q.dtype} {tuple(q.shape)}, got {t.dtype} "
                             f"{tuple(t.shape)}")
    for name, t in like_k:
        if t.shape != k.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must be {q.dtype} {tuple(k.shape)}, got {t.dtype} "
                             f"{tuple(t.shape)}")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Sq):
        raise ValueError(f"lse must be float32 {(B, Hq, Sq)}, got {lse.dtype} "
                         f"{tuple(lse.shape)}")
    if kv_lens is not None and not isinstance(kv_lens, int):
        if kv_lens.dtype != torch.int32 or tuple(kv_lens.shape) != (B, k.shape[2]):
            raise ValueError(f"kv_lens must be int32 {(B, k.shape[2])}, got "
                             f"{kv_lens.dtype} {tuple(kv_lens.shape)}")


def attn_fwd(q, k, v, o, lse, causal: bool = False, scale: float | None = None,
             kv_lens=None, stream=None) -> None:
    """O and LSE of attention. q [B,Sq,Hq,D]; k, v [B,Skv,Hkv,D]; o like q; lse [B,Hq,Sq]."""
    _check_cuda(q, k, v, o, lse, kv_lens)
    _check_shapes(q, k, v, lse, kv_lens, like_q=(("o", o),))
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    st = load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Skv,
                         D, float(scale), int(bool(causal)), _ptr(kv_lens), _dtype_code(q),
                         _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd")


def attn_fwd_paged(q, k_pages, v_pages, block_table, seq_lens, o, lse, causal: bool = False,
                   scale: float | None = None, stream=None) -> None:
    """O and LSE of attention over a paged K/V cache. q, o [B,Sq,Hq,D]; k_pages, v_pages
    [num_pages, page_size, Hkv, D]; block_table int32 [B, max_pages]; seq_lens int32 [B]
    (or None: every sequence holds max_pages * page_size keys); lse fp32 [B,Hq,Sq]."""
    _check_cuda(q, k_pages, v_pages, block_table, seq_lens, o, lse)
    if q.dim() != 4 or k_pages.dim() != 4 or v_pages.shape != k_pages.shape:
        raise ValueError("q [B,Sq,Hq,D] and page pools [pages, page_size, Hkv, D] expected")
    B, Sq, Hq, D = q.shape
    num_pages, page_size, Hkv, Dk = k_pages.shape
    if Dk != D or k_pages.dtype != q.dtype or v_pages.dtype != q.dtype:
        raise ValueError("page pools must match q in D and element type")
    if o.shape != q.shape or o.dtype != q.dtype:
        raise ValueError("o must have q's shape and element type")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Sq):
        raise ValueError(f"lse must be float32 {(B, Hq, Sq)}")
    if (block_table.dtype != torch.int32 or block_table.dim() != 2 or
            block_table.shape[0] != B):
        raise ValueError("block_table must be int32 [B, max_pages]")
    if seq_lens is not None and (seq_lens.dtype != torch.int32 or tuple(seq_lens.shape) != (B,)):
        raise ValueError("seq_lens must be int32 [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    st = load().attn_fwd_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                               _ptr(seq_lens), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, num_pages,
                               page_size, block_table.shape[1], D, float(scale),
                               int(bool(causal)), _dtype_code(q), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_paged")


def attn_fwd_splitkv_workspace_size(B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int,
                                    dtype_code: int) -> int:
    return int(load().attn_fwd_splitkv_workspace_size(B, Hq, Hkv, Sq, Skv, D, dtype_code))


def attn_fwd_splitkv(q, k, v, o, lse, causal: bool = False, scale: float | None = None,
                     kv_lens=None, workspace=None, stream=None) -> None:
    """attn_fwd for short query blocks over long K/V, with the key range split across work
    items and the partials merged. ``workspace``: a uint8 device tensor of at least
    attn_fwd_splitkv_workspace_size() bytes; allocated here (by torch) when None."""
    _check_cuda(q, k, v, o, lse, kv_lens)
    _check_shapes(q, k, v, lse, kv_lens, like_q=(("o", o),))
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    code = _dtype_code(q)
    need = attn_fwd_splitkv_workspace_size(B, Hq, Hkv, Sq, Skv, D, code)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = load().attn_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq,
                                 Skv, D, float(scale), int(bool(causal)), _ptr(kv_lens), code,
                                 _ptr(workspace), workspace.numel(), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_splitkv")


def attn_fwd_host_workspace_size(B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int,
                                 dtype_code: int) -> int:
    return int(load().attn_fwd_host_workspace_size(B, Hq, Hkv, Sq, Skv, D, dtype_code))


def attn_fwd_host(q, k, v, o, lse, causal: bool = False, scale: float | None = None,
                  kv_lens=None, workspace=None, stream=None) -> None:
    """attn_fwd on tensors in pinned host memory (q, k, v, o, lse and kv_lens CPU tensors,
    ``pin_memory()``), with the copies to and from the GPU overlapped with the compute,
    chunk by chunk of kv heads. ``workspace``: a uint8 device tensor of at least
    attn_fwd_host_workspace_size() bytes on the GPU that computes (the current device);
    allocated here (by torch) when None. Asynchronous on ``stream``: synchronise it before
    reading o and lse."""
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("lse", lse), ("kv_lens", kv_lens)):
        if t is None:
            continue
        if t.is_cuda or not t.is_pinned():
            raise ValueError(f"attn_fwd_host takes pinned host tensors ({name} is not one)")
        if not t.is_contiguous():
            raise ValueError("libattn takes contiguous tensors only")
    _check_shapes(q, k, v, lse, kv_lens, like_q=(("o", o),))
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    code = _dtype_code(q)
    need = attn_fwd_host_workspace_size(B, Hq, Hkv, Sq, Skv, D, code)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    st = load().attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Skv,
                              D, float(scale), int(bool(causal)), _ptr(kv_lens), code,
                              _ptr(workspace), workspace.numel(), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_host")


def attn_bwd_workspace_size(B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int,
                            dtype_code: int) -> int:
    return int(load().attn_bwd_workspace_size(B, Hq, Hkv, Sq, Skv, D, dtype_code))


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, causal: bool = False,
             scale: float | None = None, kv_lens=None, workspace=None, stream=None) -> None:
    """dQ, dK, dV of sum(O * dO). ``workspace``: a uint8 device tensor of at least
    attn_bwd_workspace_size() bytes; allocated here (by torch) when None."""
    _check_cuda(q, k, v, o, dout, lse, dq, dk, dv, kv_lens)
    _check_shapes(q, k, v, lse, kv_lens, like_q=(("o", o), ("dout", dout), ("dq", dq)),
                  like_k=(("dk", dk), ("dv", dv)))
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    code = _dtype_code(q)
    need = attn_bwd_workspace_size(B, Hq, Hkv, Sq, Skv, D, code)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                         _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Skv, D, float(scale),
                         int(bool(causal)), _ptr(kv_lens), code, _ptr(workspace),
                         workspace.numel(), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")


def attn_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, causal: bool = False,
                     scale: float | None = None, kv_lens=None, stream=None) -> None:
    """attn_bwd without a workspace, for callers that cannot allocate device memory: the
    scratch lives in a fixed-size array inside the library (see include/attn.h)."""
    _check_cuda(q, k, v, o, dout, lse, dq, dk, dv, kv_lens)
    _check_shapes(q, k, v, lse, kv_lens, like_q=(("o", o), ("dout", dout), ("dq", dq)),
                  like_k=(("dk", dk), ("dv", dv)))
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    st = load().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                 _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Skv, D,
                                 float(scale), int(bool(causal)), _ptr(kv_lens), _dtype_code(q),
                                 _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_noalloc")


def attn_peek_device_error(stream=None) -> tuple[int, int]:
    """(status, raw ATTN_DEVERR_* bits) of the device error word, which it clears."""
    bits = ctypes.c_uint32(0)
    st = load().attn_peek_device_error(ctypes.byref(bits), _stream(stream))
    return int(st), int(bits.value)


def forward(q, k, v, causal=False, scale=None, kv_lens=None, stream=None):
    """Allocate O and LSE (torch) and run attn_fwd."""
    B, Sq, Hq, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    attn_fwd(q, k, v, o, lse, causal, scale, kv_lens, stream)
    return o, lse


def backward(q, k, v, o, dout, lse, causal=False, scale=None, kv_lens=None, stream=None):
    """Allocate dQ, dK, dV (torch) and run attn_bwd."""
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, causal, scale, kv_lens, None, stream)
    return dq, dk, dv
