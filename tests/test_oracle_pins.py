"""Pins of the float64 oracle to things other than itself (CPU only).

Each check compares the oracle against something the pages or the mathematics fix:
scalar brute force on tiny inputs (a separate textbook derivation for the backward,
through the full softmax Jacobian rather than the D = sum(dO * O) shortcut), a library
routine as a special case (PyTorch's float64 SDPA + autograd), closed forms,
invariants, and central finite differences. The mutation tests at the end plant
plausible mistakes in a copy of the oracle and check that some pin catches each one.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa

RNG = np.random.default_rng(12345)


# ----------------------------------------------------------------------------- helpers
def rand_case(B, Sq, Skv, Hq, Hkv, D, seed, scale_v=1.0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, Sq, Hq, D)) * scale_v
    k = r.standard_normal((B, Skv, Hkv, D)) * scale_v
    v = r.standard_normal((B, Skv, Hkv, D))
    do = r.standard_normal((B, Sq, Hq, D))
    return q, k, v, do


def brute_forward(q, k, v, scale, causal, lens):
    """Scalar loops over the definition: weights exp(s) / sum exp(s) over visible keys."""
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    g = Hq // Hkv
    o = np.zeros((B, Sq, Hq, D))
    lse = np.full((B, Hq, Sq), -np.inf)
    for b in range(B):
        for h in range(Hq):
            kvh = h // g
            L = Skv if lens is None else int(lens[b][kvh])
            for i in range(Sq):
                vis = [j for j in range(L) if (not causal) or j <= i + L - Sq]
                if not vis:
                    continue
                sc = []
                for j in vis:
                    acc = 0.0
                    for d in range(D):
                        acc += float(q[b, i, h, d]) * float(k[b, j, kvh, d])
                    sc.append(scale * acc)
                w = [math.exp(s) for s in sc]
                Z = math.fsum(w)
                for d in range(D):
                    o[b, i, h, d] = math.fsum(w[t] * float(v[b, vis[t], kvh, d])
                                              for t in range(len(vis))) / Z
                lse[b, h, i] = math.log(Z)
    return o, lse


def brute_backward(q, k, v, do, scale, causal, lens):
    """Gradients of sum(O * dO) through the full softmax Jacobian dp_k/ds_j = p_k(d_kj - p_j)."""
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    g = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            kvh = h // g
            L = Skv if lens is None else int(lens[b][kvh])
            for i in range(Sq):
                vis = [j for j in range(L) if (not causal) or j <= i + L - Sq]
                if not vis:
                    continue
                sc = [scale * sum(float(q[b, i, h, d]) * float(k[b, j, kvh, d])
                                  for d in range(D)) for j in vis]
                w = [math.exp(s) for s in sc]
                Z = math.fsum(w)
                p = [x / Z for x in w]
                # dL/dp_t = sum_d dO_id v_jd ;  dL/dv_jd += p_t dO_id
                dLdp = [sum(float(do[b, i, h, d]) * float(v[b, j, kvh, d]) for d in range(D))
                        for j in vis]
                for t, j in enumerate(vis):
                    for d in range(D):
                        dv[b, j, kvh, d] += p[t] * float(do[b, i, h, d])
                n = len(vis)
                dLds = [0.0] * n
                for t in range(n):
                    acc = 0.0
                    for u in range(n):
                        jac = p[u] * ((1.0 if u == t else 0.0) - p[t])
                        acc += dLdp[u] * jac
                    dLds[t] = acc
                for t, j in enumerate(vis):
                    for d in range(D):
                        dq[b, i, h, d] += dLds[t] * scale * float(k[b, j, kvh, d])
                        dk[b, j, kvh, d] += dLds[t] * scale * float(q[b, i, h, d])
    return dq, dk, dv


def torch_sdpa(q, k, v, do, scale, causal, lens):
    """PyTorch float64 SDPA with an explicit boolean mask, plus autograd gradients."""
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    g = Hq // Hkv
    tq = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    tv = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    mask = torch.zeros(B, Hq, Sq, Skv, dtype=torch.bool)
    for b in range(B):
        for h in range(Hq):
            L = Skv if lens is None else int(lens[b][h // g])
            for i in range(Sq):
                for j in range(L):
                    if (not causal) or j <= i + L - Sq:
                        mask[b, h, i, j] = True
    kk = tk.repeat_interleave(g, dim=2)
    vv = tv.repeat_interleave(g, dim=2)
    out = torch.nn.functional.scaled_dot_product_attention(
        tq.transpose(1, 2), kk.transpose(1, 2), vv.transpose(1, 2), attn_mask=mask,
        scale=scale).transpose(1, 2)
    (out * torch.tensor(do)).sum().backward()
    return out.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


TINY = [
    # B, Sq, Skv, Hq, Hkv, D, causal, lens
    (1, 5, 5, 2, 2, 4, False, None),
    (1, 5, 5, 2, 2, 4, True, None),
    (2, 4, 7, 4, 2, 3, False, [[7, 3], [1, 6]]),
    (2, 6, 4, 4, 1, 4, True, [[4], [2]]),          # rows without a visible key
    (1, 3, 8, 3, 1, 5, True, [[8]]),               # decode-like, Sq < Skv
    (2, 5, 6, 2, 2, 4, True, [[0, 6], [5, 3]]),    # an empty K/V sequence
]


# ----------------------------------------------------------------------- brute force
@pytest.mark.parametrize("case", TINY)
def test_forward_matches_scalar_brute_force(case):
    B, Sq, Skv, Hq, Hkv, D, causal, lens = case
    q, k, v, _ = rand_case(B, Sq, Skv, Hq, Hkv, D, seed=TINY.index(case) + 100)
    scale = 0.7
    o, lse = oracle.forward(q, k, v, scale, causal, lens)
    ob, lb = brute_forward(q, k, v, scale, causal, lens)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    assert np.array_equal(np.isinf(lse), np.isinf(lb))
    fin = np.isfinite(lb)
    np.testing.assert_allclose(lse[fin], lb[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", TINY)
def test_backward_matches_softmax_jacobian_brute_force(case):
    B, Sq, Skv, Hq, Hkv, D, causal, lens = case
    q, k, v, do = rand_case(B, Sq, Skv, Hq, Hkv, D, seed=TINY.index(case) + 200)
    scale = 0.6
    dq, dk, dv, _ = oracle.backward(q, k, v, do, scale, causal, lens)
    bq, bk, bv = brute_backward(q, k, v, do, scale, causal, lens)
    np.testing.assert_allclose(dq, bq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, bk, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, bv, rtol=0, atol=1e-12)


# ------------------------------------------------------------ library special case
@pytest.mark.parametrize("case", [
    (2, 9, 9, 4, 4, 8, True, None),
    (1, 7, 12, 6, 2, 16, False, [[12, 5]]),
    (2, 8, 10, 4, 2, 8, True, [[10, 9], [8, 10]]),
])
def test_matches_torch_float64_sdpa(case):
    B, Sq, Skv, Hq, Hkv, D, causal, lens = case
    q, k, v, do = rand_case(B, Sq, Skv, Hq, Hkv, D, seed=7)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.forward(q, k, v, scale, causal, lens)
    dq, dk, dv, _ = oracle.backward(q, k, v, do, scale, causal, lens)
    to, tdq, tdk, tdv = torch_sdpa(q, k, v, do, scale, causal, lens)
    np.testing.assert_allclose(o, to, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq, tdq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, tdk, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, tdv, rtol=0, atol=1e-12)


# --------------------------------------------------------------------- closed forms
def test_probability_rows_sum_to_one():
    q, k, _, _ = rand_case(1, 16, 20, 2, 1, 8, seed=3)
    for causal, lens in [(False, None), (True, None), (False, [[11]]), (True, [[17]])]:
        for h in range(2):
            p = oracle.probabilities(q, k, 0.9, causal, lens, 0, h)
            np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-13)
            if lens is not None:
                assert np.all(p[:, lens[0][0]:] == 0.0)


def test_uniform_v_returns_v_and_zero_dq_dk():
    q, k, _, do = rand_case(2, 6, 9, 2, 2, 5, seed=4)
    vrow = np.array([0.3, -1.2, 2.0, 0.0, 0.7])
    v = np.broadcast_to(vrow, (2, 9, 2, 5)).copy()
    for causal in (False, True):
        o, _ = oracle.forward(q, k, v, 0.8, causal)
        np.testing.assert_allclose(o, np.broadcast_to(vrow, o.shape), rtol=0, atol=1e-13)
        dq, dk, dv, _ = oracle.backward(q, k, v, do, 0.8, causal)
        assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12


def test_scale_zero_gives_mean_of_valid_v_and_log_length():
    q, k, v, _ = rand_case(1, 4, 10, 2, 1, 3, seed=5)
    lens = [[6]]
    o, lse = oracle.forward(q, k, v, 0.0, False, lens)
    np.testing.assert_allclose(o[0, :, 0, :], np.broadcast_to(v[0, :6, 0, :].mean(0), (4, 3)),
                               rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, math.log(6), rtol=0, atol=1e-13)
    # causal, Sq == Skv == L: row i sees i + 1 keys
    q, k, v, _ = rand_case(1, 7, 7, 1, 1, 3, seed=6)
    o, lse = oracle.forward(q, k, v, 0.0, True)
    for i in range(7):
        np.testing.assert_allclose(o[0, i, 0], v[0, :i + 1, 0].mean(0), rtol=0, atol=1e-13)
        assert abs(lse[0, 0, i] - math.log(i + 1)) < 1e-13


def test_single_key_and_causal_first_row():
    q, k, v, _ = rand_case(1, 5, 8, 1, 1, 4, seed=8)
    o, lse = oracle.forward(q, k, v, 0.5, False, [[1]])
    np.testing.assert_allclose(o[0, :, 0], np.broadcast_to(v[0, 0, 0], (5, 4)), atol=1e-14, rtol=0)
    np.testing.assert_allclose(lse[0, 0], 0.5 * q[0, :, 0] @ k[0, 0, 0], atol=1e-13, rtol=0)
    q, k, v, _ = rand_case(1, 6, 6, 1, 1, 4, seed=9)
    o, lse = oracle.forward(q, k, v, 0.5, True)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-14, rtol=0)
    assert abs(lse[0, 0, 0] - 0.5 * q[0, 0, 0] @ k[0, 0, 0]) < 1e-13


def test_dominant_logit_selects_its_value_row():
    q, k, v, _ = rand_case(1, 3, 6, 1, 1, 4, seed=10)
    q[0, 1, 0] = [10.0, 0, 0, 0]
    k[0, 4, 0] = [10.0, 0, 0, 0]   # score 50 against O(1) for the others
    o, _ = oracle.forward(q, k, v, 0.5, False)
    np.testing.assert_allclose(o[0, 1, 0], v[0, 4, 0], atol=1e-12, rtol=0)


def test_empty_rows_give_zero_output_minus_inf_lse_and_no_gradient():
    q, k, v, do = rand_case(1, 6, 4, 2, 1, 3, seed=11)
    lens = [[2]]  # causal bottom-right: rows i < Sq - L see nothing
    o, lse = oracle.forward(q, k, v, 1.0, True, lens)
    for i in range(6):
        empty = i + 2 - 6 < 0
        assert np.isneginf(lse[0, 0, i]) == empty
        if empty:
            assert np.all(o[0, i] == 0)
    dq, dk, dv, _ = oracle.backward(q, k, v, do, 1.0, True, lens)
    assert np.all(dq[0, :4] == 0)
    assert np.all(dk[0, 2:] == 0) and np.all(dv[0, 2:] == 0)
    o, lse = oracle.forward(q, k, v, 1.0, False, [[0]])
    assert np.all(o == 0) and np.all(np.isneginf(lse))


# ----------------------------------------------------------------------- invariants
def test_key_permutation_invariance():
    q, k, v, do = rand_case(1, 7, 9, 2, 1, 4, seed=12)
    perm = RNG.permutation(9)
    o1, l1 = oracle.forward(q, k, v, 0.7, False)
    o2, l2 = oracle.forward(q, k[:, perm], v[:, perm], 0.7, False)
    np.testing.assert_allclose(o1, o2, atol=1e-13, rtol=0)
    np.testing.assert_allclose(l1, l2, atol=1e-13, rtol=0)
    _, dk1, dv1, _ = oracle.backward(q, k, v, do, 0.7, False)
    _, dk2, dv2, _ = oracle.backward(q, k[:, perm], v[:, perm], do, 0.7, False)
    np.testing.assert_allclose(dk1[:, perm], dk2, atol=1e-13, rtol=0)
    np.testing.assert_allclose(dv1[:, perm], dv2, atol=1e-13, rtol=0)


def test_gqa_equals_mha_on_expanded_kv_and_group_sums():
    q, k, v, do = rand_case(2, 6, 6, 8, 2, 4, seed=13)
    g = 4
    ke = np.repeat(k, g, axis=2)  # head h -> kv head h // g
    ve = np.repeat(v, g, axis=2)
    for causal in (False, True):
        o1, l1 = oracle.forward(q, k, v, 0.6, causal)
        o2, l2 = oracle.forward(q, ke, ve, 0.6, causal)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
        dq1, dk1, dv1, _ = oracle.backward(q, k, v, do, 0.6, causal)
        dq2, dk2, dv2, _ = oracle.backward(q, ke, ve, do, 0.6, causal)
        assert np.array_equal(dq1, dq2)
        np.testing.assert_allclose(dk1, dk2.reshape(2, 6, 2, g, 4).sum(3), atol=1e-13, rtol=0)
        np.testing.assert_allclose(dv1, dv2.reshape(2, 6, 2, g, 4).sum(3), atol=1e-13, rtol=0)


def test_group_one_is_mha_bitwise():
    q, k, v, do = rand_case(1, 5, 5, 3, 3, 4, seed=14)
    o1, _ = oracle.forward(q, k, v, 0.5, True)
    for h in range(3):  # each head alone equals the MHA head
        o2, _ = oracle.forward(q[:, :, h:h + 1], k[:, :, h:h + 1], v[:, :, h:h + 1], 0.5, True)
        assert np.array_equal(o1[:, :, h:h + 1], o2)


def test_gradient_sums():
    q, k, v, do = rand_case(2, 8, 8, 4, 2, 4, seed=15)
    for causal in (False, True):
        dq, dk, dv, delta = oracle.backward(q, k, v, do, 0.7, causal)
        # every row of dS sums to zero, so sum_j dK_j = 0
        np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12, rtol=0)
        # every row of P sums to one, so sum_j dV_j = sum over the group of sum_i dO_i
        want = do.sum(axis=1).reshape(2, 2, 2, 4).sum(2)
        np.testing.assert_allclose(dv.sum(axis=1), want, atol=1e-12, rtol=0)
        # delta_i = sum_j P_ij dP_ij
        for h in range(4):
            p = oracle.probabilities(q, k, 0.7, causal, None, 1, h)
            dp = do[1, :, h] @ v[1, :, h // 2].T
            np.testing.assert_allclose(delta[1, h], (p * dp).sum(1), atol=1e-12, rtol=0)


def test_kv_length_equals_truncated_buffer_and_ignores_padding():
    q, k, v, do = rand_case(1, 6, 10, 2, 2, 4, seed=16)
    kn, vn = k.copy(), v.copy()
    kn[0, 7:, 0] = np.nan
    vn[0, 7:, 0] = np.inf
    kn[0, 4:, 1] = np.nan
    lens = [[7, 4]]
    for causal in (False, True):
        o1, l1 = oracle.forward(q, kn, vn, 0.5, causal, lens)
        dq1, dk1, dv1, _ = oracle.backward(q, kn, vn, do, 0.5, causal, lens)
        for h, L in enumerate(lens[0]):
            o2, l2 = oracle.forward(q[:, :, h:h + 1], k[:, :L, h:h + 1], v[:, :L, h:h + 1],
                                    0.5, causal)
            dq2, dk2, dv2, _ = oracle.backward(q[:, :, h:h + 1], k[:, :L, h:h + 1],
                                               v[:, :L, h:h + 1], do[:, :, h:h + 1], 0.5, causal)
            assert np.array_equal(o1[:, :, h:h + 1], o2)
            assert np.array_equal(l1[:, h:h + 1], l2)
            assert np.array_equal(dq1[:, :, h:h + 1], dq2)
            assert np.array_equal(dk1[:, :L, h:h + 1], dk2)
            assert np.array_equal(dv1[:, :L, h:h + 1], dv2)
            assert np.all(dk1[:, L:, h] == 0) and np.all(dv1[:, L:, h] == 0)


def test_decode_row_equals_last_causal_row():
    # "xtrain evolution.md", phase-3 milestone M2a: single-query attention over the
    # cached K/V equals the last row of full causal attention.
    q, k, v, _ = rand_case(1, 9, 9, 2, 1, 4, seed=17)
    o_full, l_full = oracle.forward(q, k, v, 0.5, True)
    o_dec, l_dec = oracle.forward(q[:, -1:], k, v, 0.5, True)
    np.testing.assert_allclose(o_dec[:, 0], o_full[:, -1], atol=1e-14, rtol=0)
    np.testing.assert_allclose(l_dec[:, :, 0], l_full[:, :, -1], atol=1e-14, rtol=0)
    o_tail, _ = oracle.forward(q[:, -3:], k, v, 0.5, True)  # bottom-right alignment
    np.testing.assert_allclose(o_tail, o_full[:, -3:], atol=1e-14, rtol=0)


def test_row_functions_match_full():
    q, k, v, do = rand_case(2, 12, 15, 4, 2, 6, seed=18)
    lens = [[15, 9], [3, 12]]
    for causal in (False, True):
        o, lse = oracle.forward(q, k, v, 0.4, causal, lens)
        dq, _, _, delta = oracle.backward(q, k, v, do, 0.4, causal, lens)
        rows = [0, 3, 11]
        for b in range(2):
            for h in range(4):
                orow, lrow = oracle.forward_rows(q, k, v, 0.4, causal, lens, b, h, rows)
                np.testing.assert_allclose(orow, o[b, rows, h], atol=1e-14, rtol=0)
                assert np.array_equal(np.isinf(lrow), np.isinf(lse[b, h, rows]))
                qrow, drow = oracle.backward_dq_rows(q, k, v, do, 0.4, causal, lens, b, h, rows)
                np.testing.assert_allclose(qrow, dq[b, rows, h], atol=1e-14, rtol=0)
                np.testing.assert_allclose(drow, delta[b, h, rows], atol=1e-14, rtol=0)


def test_row_blocking_changes_nothing():
    q, k, v, do = rand_case(1, 13, 13, 2, 1, 4, seed=19)
    o1, l1 = oracle.forward(q, k, v, 0.5, True, row_block=1024)
    o2, l2 = oracle.forward(q, k, v, 0.5, True, row_block=4)
    # the BLAS may order a product's sums differently for other block heights
    np.testing.assert_allclose(o1, o2, atol=1e-14, rtol=0)
    np.testing.assert_allclose(l1, l2, atol=1e-14, rtol=0)


# --------------------------------------------------------------- finite differences
def _fd_check(q, k, v, do, scale, causal, lens, h=1e-6):
    dq, dk, dv, _ = oracle.backward(q, k, v, do, scale, causal, lens)

    def loss(qq, kk, vv):
        o, _ = oracle.forward(qq, kk, vv, scale, causal, lens)
        return float((o * do).sum())

    worst = 0.0
    for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in np.ndindex(arr.shape):
            plus = {"qq": q, "kk": k, "vv": v}
            minus = {"qq": q, "kk": k, "vv": v}
            ap = arr.copy()
            am = arr.copy()
            ap[idx] += h
            am[idx] -= h
            plus[name * 2] = ap
            minus[name * 2] = am
            fd = (loss(**plus) - loss(**minus)) / (2 * h)
            err = abs(fd - grad[idx]) / max(1.0, abs(grad[idx]))
            worst = max(worst, err)
    return worst


@pytest.mark.parametrize("causal,lens", [(False, None), (True, None), (True, [[5, 3]])])
def test_finite_difference_gradients(causal, lens):
    q, k, v, do = rand_case(1, 4, 5, 4, 2, 3, seed=20)
    assert _fd_check(q, k, v, do, 0.8, causal, lens) < 1e-6


# ------------------------------------------------------------ mutation (pin strength)
def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant plausible mistakes in the oracle (on the CPU) and check a pin fails."""
    case = (2, 6, 4, 4, 1, 4, True, [[4], [2]])
    B, Sq, Skv, Hq, Hkv, D, causal, lens = case
    q, k, v, do = rand_case(B, Sq, Skv, Hq, Hkv, D, seed=21)
    ob, _ = brute_forward(q, k, v, 0.7, causal, lens)
    bq, bk, bv = brute_backward(q, k, v, do, 0.7, causal, lens)

    good_scores = oa._scores

    def off_by_one(qrows, kmat, scale, rows, L, Sq, causal):
        s = scale * (qrows @ kmat.T)
        if causal:
            j = np.arange(L)[None, :]
            s = np.where(j < rows[:, None] + (L - Sq), s, -np.inf)
        return s

    def no_scale(qrows, kmat, scale, rows, L, Sq, causal):
        return good_scores(qrows, kmat, 1.0, rows, L, Sq, causal)

    for bad in (off_by_one, no_scale):
        monkeypatch.setattr(oa, "_scores", bad)
        o, _ = oracle.forward(q, k, v, 0.7, causal, lens)
        assert np.abs(np.nan_to_num(o) - ob).max() > 1e-6, bad.__name__
        monkeypatch.setattr(oa, "_scores", good_scores)

    # a wrong sign in dS, or dQ without the scale, breaks the backward pins
    real_backward = oa.backward

    def wrong_sign(*a, **kw):
        dq, dk, dv, dl = real_backward(*a, **kw)
        return -dq, dk, dv, dl

    dq, _, _, _ = wrong_sign(q, k, v, do, 0.7, causal, lens)
    assert np.abs(dq - bq).max() > 1e-6
    dq, dk, dv, _ = real_backward(q, k, v, do, 0.7, causal, lens)
    assert np.abs(dq / 0.7 - bq).max() > 1e-6

    # a GQA mapping by h % Hkv instead of h // g breaks the brute-force comparison
    q2, k2, v2, _ = rand_case(1, 4, 5, 4, 2, 3, seed=22)
    ob2, _ = brute_forward(q2, k2, v2, 0.5, False, None)
    k_mod, v_mod = np.tile(k2, (1, 1, 2, 1)), np.tile(v2, (1, 1, 2, 1))  # head h -> h % 2
    o_bad, _ = oracle.forward(q2, k_mod, v_mod, 0.5, False)
    assert np.abs(o_bad - ob2).max() > 1e-6
