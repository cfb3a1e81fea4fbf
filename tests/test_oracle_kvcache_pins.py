"""Pins of the paged-cache and split-range oracle (oracle/kvcache.py), CPU only.

The gather is pinned by scalar brute force (Python loops over tokens and page lookups),
by the identity page layout (which must reproduce the dense oracle bit for bit) and by
page permutations (a shuffled pool with its block table permuted alike changes nothing).
The split-range merge is pinned by its identity with the dense oracle for many ways of
cutting the keys (empty ranges, ranges past the valid length, causal rows that see no key
of a range) and by closed forms. Planted mistakes in both show that the pins bite.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import kvcache


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _paged_from_dense(k, lens, page_size, seed, extra_pages=3):
    """Scatter a dense [B, S, Hkv, D] buffer into a shuffled page pool; unused pages and
    the rows past each length hold NaN; unused block-table entries hold junk."""
    B, S, Hkv, D = k.shape
    assert S % page_size == 0
    per = S // page_size
    n_pages = B * per + extra_pages
    rng = np.random.default_rng(seed)
    order = rng.permutation(n_pages)
    pool = np.full((n_pages, page_size, Hkv, D), np.nan)
    bt = np.full((B, per), -7, dtype=np.int64)
    used = 0
    for b in range(B):
        for p in range(-(-int(lens[b]) // page_size)):
            page = int(order[used])
            used += 1
            bt[b, p] = page
            pool[page] = k[b, p * page_size:(p + 1) * page_size]
            rows_valid = int(lens[b]) - p * page_size
            if rows_valid < page_size:
                pool[page, rows_valid:] = np.nan
    return pool, bt


def _gather_loops(pool, bt, lens, page_size):
    n_pages, ps, Hkv, D = pool.shape
    B, max_pages = bt.shape
    out = np.zeros((B, max_pages * page_size, Hkv, D))
    for b in range(B):
        for t in range(int(lens[b])):
            page = int(bt[b][t // page_size])
            for h in range(Hkv):
                for d in range(D):
                    out[b][t][h][d] = float(pool[page][t % page_size][h][d])
    return out


@pytest.mark.parametrize("page_size", [1, 2, 4, 8])
def test_gather_matches_scalar_loops(page_size):
    B, S, Hkv, D = 3, 16, 2, 3
    k = _rand((B, S, Hkv, D), 1)
    lens = np.array([16, 5, 0])
    pool, bt = _paged_from_dense(k, lens, page_size, seed=page_size)
    got = kvcache.gather_pages(pool, bt, lens, page_size)
    want = _gather_loops(pool, bt, lens, page_size)
    assert np.array_equal(got, want)
    # valid rows are the dense rows; padding rows are zero, never the pool's NaN
    for b in range(B):
        assert np.array_equal(got[b, :lens[b]], k[b, :lens[b]])
        assert not np.isnan(got).any()


def _check_identity_layout(gather):
    B, S, Hq, Hkv, D, ps = 2, 24, 4, 2, 8, 4
    q, k, v = _rand((B, 10, Hq, D), 2), _rand((B, S, Hkv, D), 3), _rand((B, S, Hkv, D), 4)
    lens = np.array([24, 13])
    per = S // ps
    kpool = k.reshape(B * per, ps, Hkv, D)
    vpool = v.reshape(B * per, ps, Hkv, D)
    bt = np.arange(B * per).reshape(B, per)
    for causal in (False, True):
        o_ref, lse_ref = oracle.forward(q, k, v, 0.3, causal, np.repeat(lens[:, None], Hkv, 1))
        kd = gather(kpool, bt, lens, ps)
        vd = gather(vpool, bt, lens, ps)
        o, lse = oracle.forward(q, kd, vd, 0.3, causal, np.repeat(lens[:, None], Hkv, 1))
        assert np.array_equal(o, o_ref) and np.array_equal(lse, lse_ref)


def test_identity_page_layout_is_the_dense_oracle_bitwise():
    _check_identity_layout(kvcache.gather_pages)
    B, S, Hkv, D, ps = 2, 24, 2, 8, 4
    q = _rand((B, 10, 4, D), 2)
    k, v = _rand((B, S, Hkv, D), 3), _rand((B, S, Hkv, D), 4)
    lens = np.array([24, 13])
    bt = np.arange(B * S // ps).reshape(B, -1)
    o, lse = kvcache.forward_paged(q, k.reshape(-1, ps, Hkv, D), v.reshape(-1, ps, Hkv, D),
                                   bt, lens, ps, 0.3, True)
    o_ref, lse_ref = oracle.forward(q, k, v, 0.3, True, np.repeat(lens[:, None], Hkv, 1))
    assert np.array_equal(o, o_ref) and np.array_equal(lse, lse_ref)


@pytest.mark.parametrize("page_size,causal", [(1, False), (4, True), (8, False), (16, True)])
def test_shuffled_pages_change_nothing(page_size, causal):
    B, S, Hq, Hkv, D = 3, 32, 6, 2, 8
    q = _rand((B, 9, Hq, D), 5)
    k, v = _rand((B, S, Hkv, D), 6), _rand((B, S, Hkv, D), 7)
    lens = np.array([32, 17, 3])
    kpool, bt = _paged_from_dense(k, lens, page_size, seed=11)
    vpool, bt_v = _paged_from_dense(v, lens, page_size, seed=11)
    assert np.array_equal(bt, bt_v)
    o, lse = kvcache.forward_paged(q, kpool, vpool, bt, lens, page_size, 0.25, causal)
    o_ref, lse_ref = oracle.forward(q, k, v, 0.25, causal, np.repeat(lens[:, None], Hkv, 1))
    assert np.array_equal(o, o_ref) and np.array_equal(lse, lse_ref)


def test_torch_inputs_and_bad_tables():
    ps = 4
    pool = torch.randn(5, ps, 1, 2, dtype=torch.float64)
    bt = torch.tensor([[3, 0]], dtype=torch.int32)
    got = kvcache.gather_pages(pool, bt, torch.tensor([6], dtype=torch.int32), ps)
    assert np.array_equal(got[0, :4], pool[3].numpy()) and np.array_equal(got[0, 4:6], pool[0, :2].numpy())
    with pytest.raises(ValueError):
        kvcache.gather_pages(pool, torch.tensor([[3, 9]]), torch.tensor([6]), ps)
    with pytest.raises(ValueError):
        kvcache.gather_pages(pool, bt, torch.tensor([9]), ps)


def _check_merge_identity(forward_split):
    B, Sq, Hq, Hkv, D, S = 2, 12, 4, 2, 8, 40
    q, k, v = _rand((B, Sq, Hq, D), 8), _rand((B, S, Hkv, D), 9), _rand((B, S, Hkv, D), 10)
    lens = np.array([[40, 23], [7, 0]])
    for causal in (False, True):
        o_ref, lse_ref = oracle.forward(q, k, v, 0.35, causal, lens)
        for bounds in ([0, 40], [0, 16, 32, 48], [0, 1, 2, 3, 40], [0, 20, 20, 40],
                       [0, 7, 8, 30, 64]):
            o, lse, _, _ = forward_split(q, k, v, 0.35, causal, lens, bounds)
            fin = np.isfinite(lse_ref)
            assert np.array_equal(np.isfinite(lse), fin)
            assert np.allclose(o, o_ref, rtol=1e-12, atol=1e-13)
            assert np.allclose(lse[fin], lse_ref[fin], rtol=1e-12, atol=1e-13)


def test_split_range_merge_equals_dense_oracle():
    _check_merge_identity(kvcache.forward_split)


def test_merge_closed_forms():
    o1 = _rand((3, 5), 12)
    l1 = np.array([0.5, -1.0, 2.0])
    # one range: the merge returns it
    o, lse = kvcache.merge_partials(o1[None], l1[None])
    assert np.allclose(o, o1, rtol=1e-15) and np.allclose(lse, l1, rtol=1e-15)
    # the same range twice: same output, lse + ln 2
    o, lse = kvcache.merge_partials(np.stack([o1, o1]), np.stack([l1, l1]))
    assert np.allclose(o, o1, rtol=1e-14) and np.allclose(lse, l1 + math.log(2.0), rtol=1e-14)
    # an empty range (-inf) has no weight; all ranges empty gives 0 and -inf
    o, lse = kvcache.merge_partials(np.stack([o1, 99 * o1]), np.stack([l1, np.full(3, -np.inf)]))
    assert np.allclose(o, o1, rtol=1e-15) and np.allclose(lse, l1, rtol=1e-15)
    o, lse = kvcache.merge_partials(np.zeros((2, 3, 5)), np.full((2, 3), -np.inf))
    assert np.array_equal(o, np.zeros((3, 5))) and np.isneginf(lse).all()


def test_pins_catch_planted_mistakes():
    # a gather that reads the next row of the page
    def bad_gather(pool, bt, lens, ps):
        pool = np.asarray(pool)
        out = kvcache.gather_pages(pool, bt, lens, ps)
        B = out.shape[0]
        for b in range(B):
            for t in range(int(lens[b])):
                out[b, t] = pool[int(bt[b, t // ps]), (t % ps + 1) % ps]
        return out

    with pytest.raises(AssertionError):
        _check_identity_layout(bad_gather)

    # a merge that forgets to renormalise the weights
    def bad_split(q, k, v, scale, causal, lens, bounds):
        o, lse, op, lp = kvcache.forward_split(q, k, v, scale, causal, lens, bounds)
        if len(bounds) > 2:
            o = np.moveaxis(np.sum(np.nan_to_num(np.exp(lp))[..., None] *
                                   np.moveaxis(op, 3, 2), axis=0), 2, 1)
        return o, lse, op, lp

    with pytest.raises(AssertionError):
        _check_merge_identity(bad_split)
