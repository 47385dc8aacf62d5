"""Pins of the oracle's indexer warm-up loss (L_I = sum_t KL(p_t || softmax(I_t)),
p_t = head-aggregated dense attention, L1-normalised) and its gradient: a
closed form, the zero of the KL, library routines (softmax, kl_div), central
finite differences of the loss itself, and mutants that each must fail a pin."""

import numpy as np
import pytest
import scipy.special
import torch

import oracle


# --------------------------------------------------------------------------
# Check functions (take the implementation under test)
# --------------------------------------------------------------------------


def check_closed_form(kl_fn):
    # p uniform over n, I = (c, 0, ..., 0):
    # KL = -log n - c / n + log(e^c + n - 1)
    ok = True
    for n in (1, 2, 7, 100):
        for c in (-3.0, 0.0, 0.5, 6.0):
            p = np.full(n, 1.0 / n)
            I = np.zeros(n)
            I[0] = c
            loss, _ = kl_fn(p, I)
            want = -np.log(n) - c / n + np.log(np.exp(c) + n - 1)
            ok &= abs(loss - want) <= 1e-12 * max(1.0, abs(want))
    return bool(ok)


def check_target_against_library(target_fn):
    rng = np.random.default_rng(3)
    ok = True
    for H in (1, 3):
        Q = rng.standard_normal((H, 6))
        kv = rng.standard_normal((9, 6))
        scale = 0.4
        p = target_fn(Q, kv, scale)
        lib = scipy.special.softmax(scale * (Q @ kv.T), axis=1).mean(axis=0)
        ok &= p.shape == (9,) and abs(p.sum() - 1.0) <= 1e-14 and np.allclose(p, lib, rtol=1e-13, atol=1e-15)
    # Q = 0: every head is uniform, so is the target
    p0 = target_fn(np.zeros((4, 6)), rng.standard_normal((5, 6)), 1.0)
    ok &= np.allclose(p0, np.full(5, 0.2), rtol=0, atol=1e-15)
    return bool(ok)


def check_grad_I_by_differences(kl_fn):
    rng = np.random.default_rng(5)
    ok = True
    for n in (3, 11):
        p = rng.random(n)
        p /= p.sum()
        I = rng.standard_normal(n) * 2.0
        _, g = kl_fn(p, I)
        h = 1e-6
        fd = np.empty(n)
        for s in range(n):
            e = np.zeros(n)
            e[s] = h
            fd[s] = (kl_fn(p, I + e)[0] - kl_fn(p, I - e)[0]) / (2 * h)
        ok &= np.allclose(g, fd, rtol=1e-6, atol=1e-8)
    return bool(ok)


def _small_problem(seed=9):
    rng = np.random.default_rng(seed)
    # two sequences: a 4-token prefill and a decode query over 6 cached keys
    cu_q = np.array([0, 4, 5])
    cu_kv = np.array([0, 4, 10])
    T, S, HI, dI, H, dqk = 5, 10, 3, 4, 2, 6
    q = rng.standard_normal((T, HI, dI))
    k = rng.standard_normal((S, dI))
    w = rng.standard_normal((T, HI))
    Q = rng.standard_normal((T, H, dqk))
    kv = rng.standard_normal((S, dqk))
    return q, k, w, Q, kv, cu_q, cu_kv, 0.5


def check_input_grads_by_differences(loss_fn):
    q, k, w, Q, kv, cu_q, cu_kv, scale = _small_problem()
    _, dq, dk, dw = loss_fn(q, k, w, Q, kv, cu_q, cu_kv, scale)
    h = 1e-6

    def fd(arr, which):
        out = np.empty_like(arr)
        for ix in np.ndindex(arr.shape):
            a1, a2 = arr.copy(), arr.copy()
            a1[ix] += h
            a2[ix] -= h
            args1 = {"q": q, "k": k, "w": w}
            args2 = dict(args1)
            args1[which], args2[which] = a1, a2
            l1 = loss_fn(args1["q"], args1["k"], args1["w"], Q, kv, cu_q, cu_kv, scale)[0]
            l2 = loss_fn(args2["q"], args2["k"], args2["w"], Q, kv, cu_q, cu_kv, scale)[0]
            out[ix] = (l1 - l2) / (2 * h)
        return out

    ok = np.allclose(dq, fd(q, "q"), rtol=1e-5, atol=1e-7)
    ok &= np.allclose(dk, fd(k, "k"), rtol=1e-5, atol=1e-7)
    ok &= np.allclose(dw, fd(w, "w"), rtol=1e-5, atol=1e-7)
    return bool(ok)


# --------------------------------------------------------------------------
# Pins
# --------------------------------------------------------------------------


def test_kl_closed_form():
    assert check_closed_form(oracle.kl_to_softmax_row)


def test_kl_is_zero_at_the_target_and_positive_elsewhere():
    rng = np.random.default_rng(1)
    p = rng.random(20)
    p /= p.sum()
    loss, g = oracle.kl_to_softmax_row(p, np.log(p) + 3.25)
    assert abs(loss) <= 1e-13 and np.abs(g).max() <= 1e-13
    for _ in range(20):
        loss, _ = oracle.kl_to_softmax_row(p, rng.standard_normal(20) * 3)
        assert loss > 0


def test_kl_against_torch_kl_div():
    rng = np.random.default_rng(2)
    for n in (1, 5, 64):
        p = rng.random(n)
        p[rng.random(n) < 0.2] = 0.0          # zero-probability candidates
        if p.sum() == 0:
            p[0] = 1.0
        p /= p.sum()
        I = rng.standard_normal(n) * 4
        loss, _ = oracle.kl_to_softmax_row(p, I)
        lib = torch.nn.functional.kl_div(torch.log_softmax(torch.from_numpy(I), 0), torch.from_numpy(p),
                                         reduction="sum").item()
        assert abs(loss - lib) <= 1e-12 * max(1.0, abs(lib))


def test_target_is_the_normalised_head_sum_of_softmaxes():
    assert check_target_against_library(oracle.dense_attention_target_row)


def test_grad_wrt_scores_matches_differences():
    assert check_grad_I_by_differences(oracle.kl_to_softmax_row)


def test_grads_wrt_indexer_inputs_match_differences():
    assert check_input_grads_by_differences(oracle.indexer_warmup_loss)


def test_loss_is_the_sum_over_rows_and_uses_causal_candidates():
    q, k, w, Q, kv, cu_q, cu_kv, scale = _small_problem(seed=4)
    total = oracle.indexer_warmup_loss(q, k, w, Q, kv, cu_q, cu_kv, scale)[0]
    parts = sum(oracle.indexer_warmup_loss(q, k, w, Q, kv, cu_q, cu_kv, scale, rows=[r])[0] for r in range(5))
    assert abs(total - parts) <= 1e-12 * abs(total)
    # the first token of the prefill sees only itself: its KL is 0 whatever I is
    assert abs(oracle.indexer_warmup_loss(q, k, w, Q, kv, cu_q, cu_kv, scale, rows=[0])[0]) <= 1e-15
    # changing a key beyond a row's position leaves that row's loss unchanged
    k2 = k.copy()
    k2[3] += 5.0
    kv2 = kv.copy()
    kv2[3] += 5.0
    r2a = oracle.indexer_warmup_loss(q, k, w, Q, kv, cu_q, cu_kv, scale, rows=[2])[0]
    r2b = oracle.indexer_warmup_loss(q, k2, w, Q, kv2, cu_q, cu_kv, scale, rows=[2])[0]
    assert r2a == r2b


# --------------------------------------------------------------------------
# Mutants: each plants one plausible mistake and must fail a pin
# --------------------------------------------------------------------------


def _kl_reversed(p, I):            # KL(softmax(I) || p) instead of KL(p || softmax(I))
    q = scipy.special.softmax(I)
    pos = q > 0
    with np.errstate(divide="ignore"):
        loss = float(np.sum(q[pos] * (np.log(q[pos]) - np.log(p[pos]))))
    return loss, q - p


def _kl_grad_sign(p, I):           # gradient p - softmax(I)
    loss, g = oracle.kl_to_softmax_row(p, I)
    return loss, -g


def _target_unnormalised(Q, kv, scale):   # head sum without the L1 normalisation
    return oracle.dense_attention_target_row(Q, kv, scale) * Q.shape[0]


def _target_of_mean_scores(Q, kv, scale):  # softmax of the head-averaged scores
    return scipy.special.softmax(scale * (Q @ kv.T).mean(axis=0))


def _make_loss(backward):
    def loss_fn(q, k, w, Q, kv, cu_q, cu_kv, scale, rows=None):
        _, pos, kv0, n = oracle.query_positions(cu_q, cu_kv)
        dq, dk, dw = np.zeros_like(q), np.zeros_like(k), np.zeros_like(w)
        total = 0.0
        for r in range(len(pos)):
            a, b = kv0[r], kv0[r] + n[r]
            p = oracle.dense_attention_target_row(Q[r], kv[a:b], scale)
            I = oracle.index_scores_row(q[r], k[a:b], w[r])
            loss, g = oracle.kl_to_softmax_row(p, I)
            total += loss
            gq, gk, gw = backward(g, q[r], k[a:b], w[r])
            dq[r] += gq
            dk[a:b] += gk
            dw[r] += gw
        return total, dq, dk, dw
    return loss_fn


def _bw_no_relu_mask(g, q, k, w):
    x = q @ k.T
    dx = w[:, None] * g[None, :]
    return dx @ k, dx.T @ q, np.maximum(x, 0.0) @ g


def _bw_dk_without_w(g, q, k, w):
    dq, dk, dw = oracle.indexer_scores_backward_row(g, q, k, w)
    x = q @ k.T
    dk = ((x > 0) * g[None, :]).T @ q
    return dq, dk, dw


def test_the_reference_loss_passes_the_mutant_harness():
    assert check_input_grads_by_differences(_make_loss(oracle.indexer_scores_backward_row))


def test_mutant_reversed_kl_fails():
    assert not check_closed_form(_kl_reversed)


def test_mutant_gradient_sign_fails():
    assert not check_grad_I_by_differences(_kl_grad_sign)


@pytest.mark.parametrize("bad", [_target_unnormalised, _target_of_mean_scores])
def test_mutant_target_fails(bad):
    assert not check_target_against_library(bad)


@pytest.mark.parametrize("bad", [_bw_no_relu_mask, _bw_dk_without_w])
def test_mutant_backward_fails(bad):
    assert not check_input_grads_by_differences(_make_loss(bad))
