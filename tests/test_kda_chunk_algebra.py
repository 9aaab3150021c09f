"""The chunk algebra of Phase 2 with a decay per key channel, checked in fp64
against the per-channel oracle (``oracle.delta_fwd_kda``).

Reading of the Kimi Delta Attention backbone (section 4 of the gist.science
summary of "OSDN: Improving Delta Rule with Provable Online Preconditioning
in Linear Attention"; no formula printed there): S_t = S_{t-1} Diag(alpha_t)
+ beta_t (v_t - S_{t-1} Diag(alpha_t) k_t) ktilde_t^T, o_t = S_t q_t.  This is
the algebra a tensor-core form of it evaluates.  Within a chunk, with
Gamma_t = prod_{s <= t} alpha_s (per channel) and U the scaled residuals,

    S_t = S_0 Diag(Gamma_t) + sum_{s <= t} u_s (ktilde_s (.) Gamma_t / Gamma_s)^T

so that, with Kh = Gamma (.) K, Qh = Gamma (.) Q and Kc = Ktilde / Gamma,

    (I + tril(diag(beta) Kh Kc^T, -1)) U = diag(beta) (V - Kh S_0^T)
    O   = Qh S_0^T + tril(Qh Kc^T) U
    S_C = S_0 Diag(Gamma_C) + U^T (Ktilde (.) Gamma_C / Gamma).

1 / Gamma overflows fp32 when the decay is strong over a chunk.  The remedy
checked here takes a reference token m inside the chunk: for the pairs
s <= m <= t, Gamma_t / Gamma_s = (Gamma_t / Gamma_m) (Gamma_m / Gamma_s) with
both factors at most 1 (one product of two factored matrices); the pairs on
one side of m take the ratio Gamma_t / Gamma_s <= 1 directly (sub-chunk
blocks).  A chunk form with the decay on the value rows fails.
"""
import numpy as np
import pytest

import oracle


def chunk_kda(q, k, kt, v, beta, alpha, S0, C=64, ref_point=False, wrong_axis=False):
    T, K = k.shape
    S = S0.copy()                       # V x K
    o = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        sl = slice(c0, c0 + n)
        Q, Kk, Kt, Vc, b = q[sl], k[sl], kt[sl], v[sl], beta[sl]
        lg = np.cumsum(np.log(alpha[sl]), axis=0)          # n x K, log Gamma
        if wrong_axis:                                     # the planted mistake
            lg = lg[:, ::-1]
        if ref_point:
            m = n // 2
            gm = lg[m]                                     # log Gamma_m
            Kh, Qh = Kk * np.exp(lg - gm), Q * np.exp(lg - gm)
            Kc = Kt * np.exp(gm - lg)
            # pairs (t, s) with s <= m <= t go through m, both factors <= 1;
            # pairs on one side of m take the ratio Gamma_t / Gamma_s <= 1
            # directly (a sub-chunk block of the kernel)
            KK = np.zeros((n, n))
            QK = np.zeros((n, n))
            for t in range(n):
                for s in range(t + 1):
                    if s <= m <= t:
                        KK[t, s] = Kh[t] @ Kc[s]
                        QK[t, s] = Qh[t] @ Kc[s]
                    else:
                        r = np.exp(lg[t] - lg[s])
                        KK[t, s] = (Kk[t] * r) @ Kt[s]
                        QK[t, s] = (Q[t] * r) @ Kt[s]
            Khs = Kk * np.exp(lg)                          # S_0 terms need Gamma_t only
            Qhs = Q * np.exp(lg)
        else:
            Khs = Kk * np.exp(lg)
            Qhs = Q * np.exp(lg)
            Kc = Kt * np.exp(-lg)
            KK = Khs @ Kc.T
            QK = Qhs @ Kc.T
        L = np.tril(b[:, None] * KK, -1)
        A = np.tril(QK)
        U = np.linalg.solve(np.eye(n) + L, b[:, None] * (Vc - Khs @ S.T))
        o[sl] = Qhs @ S.T + A @ U
        gC = lg[-1]
        S = S * np.exp(gC)[None, :] + U.T @ (Kt * np.exp(gC[None, :] - lg))
    return o, S


def case(T, K, V, seed, low=0.5, high=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, K))
    k = rng.standard_normal((T, K)) / np.sqrt(K)
    kt = k * (0.5 + rng.random((T, K)))
    v = rng.standard_normal((T, V))
    beta = rng.random(T)
    alpha = low + (high - low) * rng.random((T, K))
    S0 = rng.standard_normal((V, K))
    return q, k, kt, v, beta, alpha, S0


def oracle_kda(q, k, kt, v, beta, alpha, S0):
    o, ST = oracle.delta_fwd_kda(q[None, None], k[None, None], kt[None, None], v[None, None],
                                 beta[None, None], alpha[None, None], S0[None, None])
    return o[0, 0], ST[0, 0]


@pytest.mark.parametrize("T,K,V,C", [(100, 8, 6, 64), (37, 5, 4, 16), (64, 4, 4, 64)])
def test_chunk_form_equals_recurrence(T, K, V, C):
    x = case(T, K, V, 300 + T)
    o_ref, S_ref = oracle_kda(*x)
    o, S = chunk_kda(*x, C=C)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-10 * np.abs(o_ref).max())
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-10 * np.abs(S_ref).max())


def test_reference_point_survives_strong_decay():
    # alpha in [0.1, 0.3] per token: Gamma falls below 1e-38 within a chunk,
    # so 1/Gamma overflows fp32; the reference-point form keeps every factor
    # at most 1
    x = case(64, 6, 4, 311, low=0.1, high=0.3)
    lg = np.cumsum(np.log(x[5]), axis=0)
    assert (-lg[-1]).max() / np.log(10) > 38                # 1/Gamma_C > 1e38
    o_ref, S_ref = oracle_kda(*x)
    o, S = chunk_kda(*x, C=64, ref_point=True)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-10 * np.abs(o_ref).max())
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-10 * np.abs(S_ref).max())


def test_decay_on_the_wrong_axis_fails():
    x = case(64, 6, 6, 321)
    o_ref, _ = oracle_kda(*x)
    o, _ = chunk_kda(*x, C=32, wrong_axis=True)
    assert np.abs(o - o_ref).max() > 1e-3 * np.abs(o_ref).max()
