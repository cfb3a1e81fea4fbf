"""CPU float64 oracle for attention over a paged K/V cache and over split key ranges.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may use it. It shares
no code with the CUDA library and imports nothing from the ``attention_sm_flash_gb300``
package.

Paged cache. The video-DiT's self-attention keeps its K/V in pools of fixed-size pages
that a per-sequence block table indexes, with a valid length per sequence ("LingBot
full-pipeline analysis report", section "layer-0 internal diagnosis v5": the self cache
records a block table, video slots and seq_lens, and the paged interface's key and value
pools). Its pipeline gathers the pages into contiguous K/V and runs a varlen kernel; the
report plans a direct paged kernel that reads through the block table instead (section
"optimisation migration matrix v2", row H1a_kv_gather_off: direct paged FA (block_table)
against gather + FA varlen). Both compute attention over the same keys, so the oracle
is the gather written out, followed by the dense oracle:

    token t of sequence b  =  pool[block_table[b, t // page_size], t % page_size]

for t < seq_lens[b]; positions at or past seq_lens[b] are padding (never read here, and
masked by the valid length like any varlen padding).

Split key ranges. Attention over a key set that is the disjoint union of ranges R_s is
the merge of the attentions over each range: with O_s, lse_s the normalised output and
log-sum-exp over R_s alone, lse = log(sum_s exp(lse_s)) and O = sum_s exp(lse_s - lse) O_s
(a range with no visible key has lse_s = -inf and weight 0). This is the identity a
split-KV forward relies on when short query blocks (single-query decode, "xtrain
evolution.md", phase-3 milestone M2a: decode attention = the last causal row) are spread
over many key ranges; ``forward_split`` computes it step by step so that the identity
itself is pinned against the dense oracle.

Parity status: every public function here is pinned by the CPU tests (scalar brute force
of the gather, identity and permuted page layouts against the dense oracle, the merge
identity, planted mistakes); none is "parity unpinned".
"""

from __future__ import annotations

import numpy as np

from .attention import _f64, _scores, _softmax_rows, forward

__all__ = ["gather_pages", "forward_paged", "merge_partials", "forward_split"]


def _ints(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.asarray(x, dtype=np.int64)


def gather_pages(pool, block_table, seq_lens, page_size: int) -> np.ndarray:
    """Contiguous K (or V) [B, max_pages * page_size, Hkv, D] from a paged pool.

    ``pool``: [num_pages, page_size, Hkv, D]; ``block_table``: int [B, max_pages];
    ``seq_lens``: int [B]. Rows at or past a sequence's length are zero (padding), and
    block-table entries of pages that hold no valid token are never read.
    """
    pool = _f64(pool)
    bt = _ints(block_table)
    lens = _ints(seq_lens).reshape(-1)
    num_pages, ps, Hkv, D = pool.shape
    if ps != page_size:
        raise ValueError("pool's second dimension must be the page size")
    B, max_pages = bt.shape
    smax = max_pages * page_size
    if lens.shape[0] != B or (lens < 0).any() or (lens > smax).any():
        raise ValueError("seq_lens must be [B] with entries in [0, max_pages * page_size]")
    out = np.zeros((B, smax, Hkv, D))
    for b in range(B):
        L = int(lens[b])
        for t0 in range(0, L, page_size):
            page = int(bt[b, t0 // page_size])
            if page < 0 or page >= num_pages:
                raise ValueError(f"block_table[{b}, {t0 // page_size}] = {page} is not a page")
            n = min(page_size, L - t0)
            out[b, t0:t0 + n] = pool[page, :n]
    return out


def forward_paged(q, k_pool, v_pool, block_table, seq_lens, page_size: int, scale: float,
                  causal: bool = False):
    """Attention of q [B, Sq, Hq, D] over the paged K/V of each sequence: the gather
    above, then the dense oracle with every kv head's valid length = seq_lens[b].

    Returns ``(o [B,Sq,Hq,D], lse [B,Hq,Sq])``."""
    k = gather_pages(k_pool, block_table, seq_lens, page_size)
    v = gather_pages(v_pool, block_table, seq_lens, page_size)
    B, _, Hkv, _ = k.shape
    lens = np.repeat(_ints(seq_lens).reshape(B, 1), Hkv, axis=1)
    return forward(q, k, v, scale, causal, lens)


def merge_partials(o_parts, lse_parts):
    """Merge normalised partial attentions over disjoint key ranges.

    ``o_parts`` [n, ..., D] and ``lse_parts`` [n, ...]: range s's output and natural-log
    LSE (-inf where the range holds no visible key). Returns (o [..., D], lse [...]);
    rows with no visible key in any range give o = 0, lse = -inf."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = np.max(lse_parts, axis=0)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    w = np.exp(lse_parts - m_safe[None])  # exp(-inf) = 0 for empty ranges
    total = w.sum(axis=0)
    lse = np.full(m.shape, -np.inf)
    lse[has] = m_safe[has] + np.log(total[has])
    wn = np.zeros_like(w)
    wn[:, has] = w[:, has] / total[has][None]
    o = np.sum(wn[..., None] * o_parts, axis=0)
    return o, lse


def forward_split(q, k, v, scale: float, causal: bool, kv_lens, bounds):
    """The forward computed as separate attentions over the key ranges
    [bounds[s], bounds[s + 1]) and merged with :func:`merge_partials`.

    ``bounds``: increasing key positions from 0 to at least Skv. Masks (valid length,
    causal bottom-right) are those of the whole problem. Returns (o, lse, o_parts,
    lse_parts) with the partials [n, B, Sq, Hq, D] and [n, B, Hq, Sq]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, Hq, D = q.shape
    _, Skv, Hkv, _ = k.shape
    g = Hq // Hkv
    lens = (np.full((B, Hkv), Skv, dtype=np.int64) if kv_lens is None
            else _ints(kv_lens).reshape(B, Hkv))
    n = len(bounds) - 1
    o_parts = np.zeros((n, B, Sq, Hq, D))
    lse_parts = np.full((n, B, Hq, Sq), -np.inf)
    rows = np.arange(Sq)
    for b in range(B):
        for h in range(Hq):
            kvh = h // g
            L = int(lens[b, kvh])
            s_full = _scores(q[b, :, h, :], k[b, :L, kvh, :], scale, rows, L, Sq, causal)
            for sidx in range(n):
                j0, j1 = min(bounds[sidx], L), min(bounds[sidx + 1], L)
                p, m, l, has = _softmax_rows(s_full[:, j0:j1])
                o_parts[sidx, b, :, h, :] = p @ v[b, j0:j1, kvh, :]
                lse_parts[sidx, b, h, has] = m[has] + np.log(l[has])
    o_m, lse_m = merge_partials(np.moveaxis(o_parts, 3, 2), lse_parts)
    return np.moveaxis(o_m, 2, 1), lse_m, o_parts, lse_parts
