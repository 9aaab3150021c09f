"""Pins for the per-channel-decay oracle (``oracle.delta_fwd_kda``,
``oracle.forward_kda``): the Kimi Delta Attention backbone named in section 4
of the gist.science summary of "OSDN: Improving Delta Rule with Provable
Online Preconditioning in Linear Attention", read as a decay per key channel
in place of the scalar gate of the Gated DeltaNet backbone (the pages print
no formula for either):

    S_t = S_{t-1} Diag(alpha_t) + beta_t (v_t - S_{t-1} Diag(alpha_t) k_t) ktilde_t^T
    o_t = S_t q_t

Each pin fixes the result by something other than the oracle's own loop:

(1) the transition-matrix form S_t = S_{t-1} Diag(alpha_t) (I - beta_t k_t
    ktilde_t^T) + beta_t v_t ktilde_t^T, evaluated with dense matrix products;
(2) a token with alpha_t = 0 resets the state to beta_t v_t ktilde_t^T;
(3) one-hot keys decouple the key columns: column j is a scalar recurrence
    with the closed form sum_t beta_t v_t prod_{u > t} c_uj + prod_t c_tj S0,
    c_tj = alpha_tj (1 - beta_t) if token t writes column j, else alpha_tj;
(4) equal channels give the scalar-gated oracle (itself pinned elsewhere);
(5) the autograd reference with a per-channel decay equals the C oracle's
    forward and its gradients equal finite differences of it;
(6) a stored fixture of (3) in exact rationals (tests/golden/, written by a
    closed-form script that calls no oracle).

A decay applied along the value rows instead of the key columns fails (1).
"""
import numpy as np
import pytest

import oracle
from oracle import backward


def rand_case(T, K, V, seed, reset_at=None):
    rng = np.random.default_rng(seed)
    B, H = 1, 2
    q = rng.standard_normal((B, H, T, K))
    k = rng.standard_normal((B, H, T, K)) / np.sqrt(K)
    kt = k * (0.5 + rng.random((B, H, T, K)))
    v = rng.standard_normal((B, H, T, V))
    beta = rng.random((B, H, T))
    alpha = 0.5 + 0.5 * rng.random((B, H, T, K))
    if reset_at is not None:
        alpha[:, :, reset_at] = 0.0
    S0 = rng.standard_normal((B, H, V, K))
    return q, k, kt, v, beta, alpha, S0


def transition_form(q, k, kt, v, beta, alpha, S0, decay_rows=False):
    T, K = k.shape
    S = S0.copy()
    o = np.zeros((T, v.shape[1]))
    for t in range(T):
        if decay_rows:   # the planted mistake: decay the value rows
            Dk = np.eye(K)
            S = np.diag(alpha[t][: S.shape[0]]) @ S if S.shape[0] <= K else S
        else:
            Dk = np.diag(alpha[t])
        S = S @ Dk @ (np.eye(K) - beta[t] * np.outer(k[t], kt[t])) + beta[t] * np.outer(v[t], kt[t])
        o[t] = S @ q[t]
    return o, S


@pytest.mark.parametrize("T,K,V", [(11, 5, 3), (16, 4, 6), (1, 3, 2)])
def test_pin_transition_matrix_form(T, K, V):
    q, k, kt, v, beta, alpha, S0 = rand_case(T, K, V, 10 + T)
    o, ST = oracle.delta_fwd_kda(q, k, kt, v, beta, alpha, S0)
    for h in range(2):
        o_m, S_m = transition_form(q[0, h], k[0, h], kt[0, h], v[0, h], beta[0, h], alpha[0, h],
                                   S0[0, h])
        np.testing.assert_allclose(o[0, h], o_m, rtol=0, atol=1e-12 * max(1, np.abs(o_m).max()))
        np.testing.assert_allclose(ST[0, h], S_m, rtol=0, atol=1e-12 * max(1, np.abs(S_m).max()))


def test_pin_catches_a_decay_on_the_wrong_axis():
    q, k, kt, v, beta, alpha, S0 = rand_case(9, 5, 3, 31)
    o, _ = oracle.delta_fwd_kda(q, k, kt, v, beta, alpha, S0)
    o_bad, _ = transition_form(q[0, 0], k[0, 0], kt[0, 0], v[0, 0], beta[0, 0], alpha[0, 0],
                               S0[0, 0], decay_rows=True)
    assert np.abs(o[0, 0] - o_bad).max() > 1e-3 * np.abs(o[0, 0]).max()


def test_pin_zero_decay_resets_the_state():
    T, K, V, r = 7, 6, 4, 4
    q, k, kt, v, beta, alpha, S0 = rand_case(T, K, V, 41, reset_at=r)
    o, _ = oracle.delta_fwd_kda(q[:, :, : r + 1], k[:, :, : r + 1], kt[:, :, : r + 1],
                                v[:, :, : r + 1], beta[:, :, : r + 1], alpha[:, :, : r + 1], S0)
    for h in range(2):
        S_r = beta[0, h, r] * np.outer(v[0, h, r], kt[0, h, r])
        np.testing.assert_allclose(o[0, h, r], S_r @ q[0, h, r], rtol=0, atol=1e-13)


def test_pin_one_hot_keys_closed_form():
    rng = np.random.default_rng(51)
    T, K, V = 20, 6, 3
    cols = rng.integers(0, K, T)
    k = np.zeros((1, 1, T, K))
    k[0, 0, np.arange(T), cols] = 1.0
    q = rng.standard_normal((1, 1, T, K))
    v = rng.standard_normal((1, 1, T, V))
    beta = rng.random((1, 1, T))
    alpha = 0.3 + 0.7 * rng.random((1, 1, T, K))
    S0 = rng.standard_normal((1, 1, V, K))
    _, ST = oracle.delta_fwd_kda(q, k, k, v, beta, alpha, S0)
    a, b = alpha[0, 0], beta[0, 0]
    c = a.copy()
    c[np.arange(T), cols] *= 1.0 - b
    want = np.zeros((V, K))
    for j in range(K):
        tail = np.append(np.cumprod(c[::-1, j])[::-1], 1.0)     # tail[t] = prod_{u >= t} c_uj
        want[:, j] = tail[0] * S0[0, 0, :, j]
        for t in np.nonzero(cols == j)[0]:
            want[:, j] += b[t] * v[0, 0, t] * tail[t + 1]
    np.testing.assert_allclose(ST[0, 0], want, rtol=0, atol=1e-13)


def test_equal_channels_give_the_scalar_gate():
    q, k, kt, v, beta, alpha, S0 = rand_case(13, 4, 5, 61)
    a = alpha[..., 0]
    o1, S1 = oracle.delta_fwd(q, k, kt, v, beta, a, S0)
    o2, S2 = oracle.delta_fwd_kda(q, k, kt, v, beta, np.repeat(a[..., None], 4, -1), S0)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


def test_autograd_reference_matches_and_differentiates_the_kda_oracle():
    rng = np.random.default_rng(71)
    B, H, T, K, V = 1, 1, 6, 4, 3
    q, k, kt_unused, v, beta, alpha, S0 = rand_case(T, K, V, 72)
    q, k, v, beta, alpha, S0 = (x[:, :1] for x in (q, k, v, beta, alpha, S0))
    r = 0.8 + 0.2 * rng.random((B, H, T))
    d0 = 0.5 + rng.random((B, H, K))
    eta = 0.1
    ref = oracle.forward_kda(q, k, v, beta, r, eta, d0, alpha, S0)
    t = {n: backward._t(x) for n, x in dict(q=q, k=k, v=v, beta=beta, r=r, d0=d0, alpha=alpha,
                                             S0=S0).items()}
    got = backward.forward_torch(t["q"], t["k"], t["v"], t["beta"], t["r"], eta, t["d0"],
                                 t["alpha"], t["S0"])
    for gt, rf in zip(got, ref):
        np.testing.assert_allclose(gt.numpy(), rf, rtol=0, atol=1e-12 * max(1, np.abs(rf).max()))
    do = rng.standard_normal((B, H, T, V))
    dST = rng.standard_normal((B, H, V, K))
    g = backward.grads(q, k, v, beta, r, eta, d0, alpha, S0, do=do, dST=dST)

    def loss(a, s):
        _, _, o, ST = oracle.forward_kda(q, k, v, beta, r, eta, d0, a, s, nthreads=1)
        return np.sum(o * do) + np.sum(ST * dST)

    h = 1e-6
    for name, base in (("alpha", alpha), ("S0", S0)):
        num = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            p, m = base.copy(), base.copy()
            p[idx] += h
            m[idx] -= h
            args_p = (p, S0) if name == "alpha" else (alpha, p)
            args_m = (m, S0) if name == "alpha" else (alpha, m)
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(g[name], num, rtol=0, atol=1e-6 * max(1, np.abs(num).max()),
                                   err_msg=name)


def test_golden_one_hot_fixture():
    # exact rationals from tests/golden/make_kda_one_hot_fixture.py (closed
    # form, no oracle call)
    import os
    from fractions import Fraction
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "kda_one_hot_closed_form.txt")
    vals = {}
    for line in open(path):
        if line.startswith("#") or "=" not in line:
            continue
        key, rhs = (s.strip() for s in line.split("=", 1))
        vals[key] = [float(Fraction(x)) for x in rhs.split()]
    K, V = int(vals["K"][0]), int(vals["V"][0])
    cols = [int(c) for c in vals["cols"]]
    T = len(cols)
    k = np.zeros((1, 1, T, K))
    k[0, 0, np.arange(T), cols] = 1.0
    q = np.array([vals["q_%d" % t] for t in range(T)])[None, None]
    v = np.array([vals["v_%d" % t] for t in range(T)])[None, None]
    alpha = np.array([vals["alpha_%d" % t] for t in range(T)])[None, None]
    beta = np.array(vals["beta"])[None, None]
    S0 = np.array([vals["S0_%d" % i] for i in range(V)])[None, None]
    o, ST = oracle.delta_fwd_kda(q, k, k, v, beta, alpha, S0)
    np.testing.assert_allclose(o[0, 0], np.array([vals["o_%d" % t] for t in range(T)]),
                               rtol=0, atol=1e-14)
    np.testing.assert_allclose(ST[0, 0], np.array([vals["ST_%d" % i] for i in range(V)]),
                               rtol=0, atol=1e-14)
