"""CPU float64 oracle for scaled-dot-product attention (forward and backward).

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call or run this
module: only the test suite, the smoke check in ``__graft_entry__`` and the CPU-baseline
leg of ``bench.py`` use it. It shares no code with the CUDA library and imports nothing
from the ``attention_sm_flash_gb300`` package.

What it computes is the plain, composed definition of attention: materialise the score
matrix, mask it, take an exact (two-pass, full-row) softmax, multiply by V. A fused
"flash" kernel is an exact reformulation of this same result (online softmax over K/V
tiles, never materialising the N x N scores), so the definition itself is the oracle:

* "xtrain evolution.md", infra table, row T4: attention composed from matmul + softmax,
  the parity target the fused kernel is checked against;
* same table, row T14 (fused flash attention): forward = online softmax tiled over K/V;
  backward recomputes the scores and uses D = sum(dO * O) to simplify the softmax
  Jacobian, producing dQ, dK, dV;
* same table, row T15 (true GQA): K/V are broadcast to the query heads with
  ``dst = kvh * group + r`` (query head h reads kv head h // group), and the backward of
  that broadcast is a deterministic in-group sum of the query heads' gradients;
* "LingBot full-pipeline analysis report", section "Attention: real inputs, backends,
  errors and timing": the FP64 reference covers all *valid* K/V; section "same-GPU
  FA2/FA3 hardware comparison": K/V storage past the valid (cu_seqlens) length is
  padding and must not enter the reference;
* same report, section "memory boundary of long-KV at high resolution": the composed
  "math" path materialises a dense H x Q x K score matrix, which is why this oracle
  works in row blocks (each row's arithmetic is the same in any blocking, up to the
  summation order the BLAS picks for a product).

Conventions (the pages leave these open; the readings are stated here and listed with
the rest of the design):

* layout: q, o, do, dq are [B, Sq, Hq, D]; k, v, dk, dv are [B, Skv, Hkv, D];
  lse and delta are [B, Hq, Sq];
* ``kv_lens``: optional int array [B, Hkv]; keys j >= kv_lens[b, kvh] are invalid;
  ``None`` means every length is Skv;
* causal: bottom-right aligned, key j is visible to query i iff j <= i + (L - Sq),
  L the valid key length. With Sq == Skv == L this is the usual j <= i;
* scale multiplies q.k before the mask and the softmax;
* lse = natural log of sum over valid keys of exp(scale * q.k);
* a query row with no valid key has O = 0, lse = -inf and contributes no gradient.

Parity status: every public function here is pinned by the CPU tests (scalar brute
force, a library routine as a special case, closed forms, invariants and finite
differences); none is "parity unpinned".
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "forward",
    "backward",
    "probabilities",
    "forward_rows",
    "backward_dq_rows",
    "valid_length",
]

ROW_BLOCK = 1024  # rows of the score matrix materialised at once (memory only)


def _f64(x) -> np.ndarray:
    """Upcast an array-like (numpy or torch CPU tensor) to a float64 numpy array."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        try:
            import torch  # local: torch is optional for the oracle itself

            x = x.to(torch.float64)
        except Exception:  # pragma: no cover
            pass
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def _lens(kv_lens, B: int, Hkv: int, Skv: int) -> np.ndarray:
    """Valid key lengths as an int64 [B, Hkv] array (``None`` -> all Skv)."""
    if kv_lens is None:
        return np.full((B, Hkv), Skv, dtype=np.int64)
    if hasattr(kv_lens, "detach"):
        kv_lens = kv_lens.detach().to("cpu").numpy()
    lens = np.asarray(kv_lens, dtype=np.int64).reshape(B, Hkv)
    if (lens < 0).any() or (lens > Skv).any():
        raise ValueError("kv_lens entries must lie in [0, Skv]")
    return lens


def valid_length(kv_lens, b: int, kvh: int, B: int, Hkv: int, Skv: int) -> int:
    """The number of valid keys of (batch b, kv head kvh)."""
    return int(_lens(kv_lens, B, Hkv, Skv)[b, kvh])


def _scores(qrows: np.ndarray, kmat: np.ndarray, scale: float, rows: np.ndarray,
            L: int, Sq: int, causal: bool) -> np.ndarray:
    """Masked scaled scores for the given query row indices against the L valid keys.

    Returns [len(rows), L] float64 with -inf at masked positions.
    """
    s = scale * (qrows @ kmat.T)
    if causal:
        # key j is visible to query i iff j <= i + (L - Sq)
        j = np.arange(L)[None, :]
        limit = rows[:, None] + (L - Sq)
        s = np.where(j <= limit, s, -np.inf)
    return s


def _softmax_rows(s: np.ndarray):
    """Exact two-pass softmax of each row; rows with no finite entry give zeros.

    Returns (P normalised, m row max, l row sum of exp(s - m)).
    """
    m = np.max(s, axis=1) if s.shape[1] > 0 else np.full(s.shape[0], -np.inf)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    e = np.exp(s - m_safe[:, None])  # exp(-inf) = 0 on masked entries
    e[~has] = 0.0
    l = e.sum(axis=1)
    p = np.zeros_like(e)
    p[has] = e[has] / l[has, None]
    return p, m, l, has


def probabilities(q, k, scale: float, causal: bool = False, kv_lens=None,
                  b: int = 0, h: int = 0) -> np.ndarray:
    """Normalised attention probabilities P[Sq, Skv] of one (b, h); invalid keys are 0."""
    q = _f64(q)
    k = _f64(k)
    B, Sq, Hq, D = q.shape
    _, Skv, Hkv, _ = k.shape
    g = Hq // Hkv
    kvh = h // g
    L = valid_length(kv_lens, b, kvh, B, Hkv, Skv)
    rows = np.arange(Sq)
    s = _scores(q[b, :, h, :], k[b, :L, kvh, :], scale, rows, L, Sq, causal)
    p, _, _, _ = _softmax_rows(s)
    out = np.zeros((Sq, Skv))
    out[:, :L] = p
    return out


def _check_shapes(q, k, v):
    B, Sq, Hq, D = q.shape
    Bk, Skv, Hkv, Dk = k.shape
    if v.shape != k.shape or Bk != B or Dk != D:
        raise ValueError("q [B,Sq,Hq,D], k and v [B,Skv,Hkv,D] expected")
    if Hkv == 0 or Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return B, Sq, Hq, D, Skv, Hkv, Hq // Hkv


def forward(q, k, v, scale: float, causal: bool = False, kv_lens=None,
            row_block: int = ROW_BLOCK):
    """O = softmax(mask(scale * Q K^T)) V and the row log-sum-exp, in float64.

    Returns ``(o [B,Sq,Hq,D], lse [B,Hq,Sq])``.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, Hq, D, Skv, Hkv, g = _check_shapes(q, k, v)
    lens = _lens(kv_lens, B, Hkv, Skv)
    o = np.zeros((B, Sq, Hq, D))
    lse = np.full((B, Hq, Sq), -np.inf)
    for b in range(B):
        for h in range(Hq):
            kvh = h // g  # GQA: query head h reads kv head h // g
            L = int(lens[b, kvh])
            kmat = k[b, :L, kvh, :]
            vmat = v[b, :L, kvh, :]
            for i0 in range(0, Sq, row_block):
                rows = np.arange(i0, min(Sq, i0 + row_block))
                s = _scores(q[b, rows, h, :], kmat, scale, rows, L, Sq, causal)
                p, m, l, has = _softmax_rows(s)
                o[b, rows, h, :] = p @ vmat
                lse[b, h, rows[has]] = m[has] + np.log(l[has])
    return o, lse


def backward(q, k, v, do, scale: float, causal: bool = False, kv_lens=None,
             row_block: int = ROW_BLOCK):
    """Analytic gradients of sum(O * dO) with respect to Q, K and V, in float64.

    With P the normalised probabilities of the valid keys:
    dV = P^T dO; dP = dO V^T; delta_i = sum_d dO_id O_id; dS = P * (dP - delta);
    dQ = scale dS K; dK = scale dS^T Q. The kv-head gradients are summed over the
    query heads of their group; invalid keys get zero gradient.

    Returns ``(dq, dk, dv, delta)`` with delta [B, Hq, Sq].
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Sq, Hq, D, Skv, Hkv, g = _check_shapes(q, k, v)
    if do.shape != q.shape:
        raise ValueError("do must have the shape of q")
    lens = _lens(kv_lens, B, Hkv, Skv)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    delta = np.zeros((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            kvh = h // g
            L = int(lens[b, kvh])
            kmat = k[b, :L, kvh, :]
            vmat = v[b, :L, kvh, :]
            for i0 in range(0, Sq, row_block):
                rows = np.arange(i0, min(Sq, i0 + row_block))
                qr = q[b, rows, h, :]
                dor = do[b, rows, h, :]
                s = _scores(qr, kmat, scale, rows, L, Sq, causal)
                p, _, _, _ = _softmax_rows(s)
                o_r = p @ vmat
                dlt = np.sum(dor * o_r, axis=1)
                delta[b, h, rows] = dlt
                dp = dor @ vmat.T
                ds = p * (dp - dlt[:, None])
                dq[b, rows, h, :] = scale * (ds @ kmat)
                dk[b, :L, kvh, :] += scale * (ds.T @ qr)
                dv[b, :L, kvh, :] += p.T @ dor
    return dq, dk, dv, delta


def forward_rows(q, k, v, scale: float, causal: bool, kv_lens, b: int, h: int, rows):
    """Forward output rows of one (b, h): returns (o [n, D], lse [n]) for query ``rows``.

    The same arithmetic as :func:`forward`, restricted to some rows, so that a sample of
    a large problem can be checked one row at a time.
    """
    q, k, v = _f64(q[b:b + 1]), _f64(k[b:b + 1]), _f64(v[b:b + 1])
    _, Sq, Hq, D = q.shape
    _, Skv, Hkv, _ = k.shape
    g = Hq // Hkv
    kvh = h // g
    L = _row_len(kv_lens, b, kvh, Hkv, Skv)
    rows = np.asarray(rows, dtype=np.int64)
    s = _scores(q[0, rows, h, :], k[0, :L, kvh, :], scale, rows, L, Sq, causal)
    p, m, l, has = _softmax_rows(s)
    o = p @ v[0, :L, kvh, :]
    lse = np.full(len(rows), -np.inf)
    lse[has] = m[has] + np.log(l[has])
    return o, lse


def _row_len(kv_lens, b: int, kvh: int, Hkv: int, Skv: int) -> int:
    if kv_lens is None:
        return Skv
    if hasattr(kv_lens, "detach"):
        kv_lens = kv_lens.detach().to("cpu").numpy()
    lens = np.asarray(kv_lens, dtype=np.int64).reshape(-1, Hkv)
    L = int(lens[b, kvh])
    if L < 0 or L > Skv:
        raise ValueError("kv_lens entries must lie in [0, Skv]")
    return L


def backward_dq_rows(q, k, v, do, scale: float, causal: bool, kv_lens, b: int, h: int,
                     rows):
    """dQ rows of one (b, h) (and their delta), computed from those rows alone."""
    q, k, v, do = _f64(q[b:b + 1]), _f64(k[b:b + 1]), _f64(v[b:b + 1]), _f64(do[b:b + 1])
    _, Sq, Hq, D = q.shape
    _, Skv, Hkv, _ = k.shape
    g = Hq // Hkv
    kvh = h // g
    L = _row_len(kv_lens, b, kvh, Hkv, Skv)
    rows = np.asarray(rows, dtype=np.int64)
    kmat = k[0, :L, kvh, :]
    vmat = v[0, :L, kvh, :]
    s = _scores(q[0, rows, h, :], kmat, scale, rows, L, Sq, causal)
    p, _, _, _ = _softmax_rows(s)
    dor = do[0, rows, h, :]
    o_r = p @ vmat
    dlt = np.sum(dor * o_r, axis=1)
    ds = p * (dor @ vmat.T - dlt[:, None])
    return scale * (ds @ kmat), dlt
