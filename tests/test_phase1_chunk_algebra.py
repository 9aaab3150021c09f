"""The chunk algebra the Phase 1 kernels evaluate, checked in fp64.

The scan kernels do not step d token by token through a K-wide reduction:
per chunk of 16 tokens starting from d, with w_t = k_t (.) k_t,
n_t = ||k_t||^2, c_t = eta beta_t / n_t, p_t = <d, w_t>, G_tu = <w_t, w_u>,
rho_t = prod_{v<t} r_v and pi_ut = prod_{u<v<t} r_v, they use

    <d_t, w_t> = rho_t p_t + sum_{u<t} pi_ut e_u G_tu,
    e_t        = c_t (1 - beta_t <d_t, w_t>)

so the 16 step sizes e_t of a chunk come from one lower-triangular
substitution, e_t = c_t - c_t beta_t rho_t p_t - sum_{u<t} coef_tu e_u with
coef_tu = c_t beta_t pi_ut G_tu, after which every column of d steps through
the chunk on its own (ktilde_t = d_t (.) k_t, d_{t+1} = r_t d_t + e_t w_t).
The residual factor of the diagnostic is y_t = 1 - beta_t <d_t, w_t>
= 1 - beta_t rho_t p_t - sum_u beta_t pi_ut G_tu e_u.

This test restates that algebra in plain fp64 numpy and compares it with the
oracle's token recurrence (gist.science summary of arXiv 2605.13473,
sections 2.2 and 2.3); a dropped retention factor must fail it.
"""
import numpy as np
import pytest

import oracle
from preconditioned_delta_rule_phase1_gb300 import synth


def chunk_scan(k, beta, r, eta, d0, C=16, drop_pi=False):
    """Phase 1 for one sequence by the per-chunk algebra above (fp64)."""
    T, K = k.shape
    d = np.ones(K) if d0 is None else d0.astype(np.float64).copy()
    kt = np.zeros((T, K))
    lr = 0.0
    rr_all = np.ones(T) if r is None else r
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        kc, b, rr = k[c0:c0 + n], beta[c0:c0 + n], rr_all[c0:c0 + n]
        w = kc * kc
        nn = w.sum(axis=1)
        c = np.where(nn > 0, eta * b / np.where(nn > 0, nn, 1.0), 0.0)
        p = w @ d
        G = w @ w.T
        rho = np.concatenate([[1.0], np.cumprod(rr)[:-1]])           # prod_{v<t} r_v
        pi = np.ones((n, n))
        if not drop_pi:
            for t in range(n):
                for u in range(t):
                    pi[t, u] = np.prod(rr[u + 1:t])
        e = np.zeros(n)
        y = np.zeros(n)
        for t in range(n):
            s = sum(pi[t, u] * G[t, u] * e[u] for u in range(t))
            a_t = rho[t] * p[t] + s
            e[t] = c[t] * (1.0 - b[t] * a_t)
            y[t] = 1.0 - b[t] * a_t
        for t in range(n):
            kt[c0 + t] = d * kc[t]
            d = rr[t] * d + e[t] * w[t]
        lr += float(np.sum(np.log(y * y)))
    return kt, d, lr


@pytest.mark.parametrize("T,apf,seed", [(16, True, 1), (100, True, 2), (77, False, 3), (203, True, 4)])
def test_phase1_chunk_algebra_equals_token_recurrence(T, apf, seed):
    x = synth.make_random(1, 2, T, 24, 8, io="f32", apf=apf, d0=True, seed=seed)
    f64 = lambda t: None if t is None else t.double().numpy()
    k, beta, r, d0 = f64(x["k"]), f64(x["beta"]), f64(x["r"]), f64(x["d0"])
    okt, odT, olr = oracle.precond_scan(k, beta, r, x["eta"], d0, log_ratio=True)
    for h in range(2):
        kt, dT, lr = chunk_scan(k[0, h], beta[0, h], None if r is None else r[0, h], x["eta"],
                                d0[0, h])
        np.testing.assert_allclose(kt, okt[0, h], rtol=0, atol=1e-12 * np.abs(kt).max())
        np.testing.assert_allclose(dT, odT[0, h], rtol=0, atol=1e-12 * np.abs(dT).max())
        assert abs(lr - olr[0, h]) <= 1e-10 * max(1.0, abs(lr))


def test_phase1_chunk_algebra_catches_a_dropped_retention_factor():
    # the same algebra with pi_ut = 1 (retention left out of the coupling)
    # must not pass: the comparison above is sensitive to the r terms
    x = synth.make_random(1, 1, 64, 24, 8, io="f32", apf=True, seed=9)
    x["r"] = x["r"] * 0.5    # strong retention, so the coupling term matters
    x["eta"] = 2.0
    f64 = lambda t: None if t is None else t.double().numpy()
    k, beta, r = f64(x["k"]), f64(x["beta"]), f64(x["r"])
    okt, _ = oracle.precond_scan(k, beta, r, x["eta"], None)
    kt, _, _ = chunk_scan(k[0, 0], beta[0, 0], r[0, 0], x["eta"], None, drop_pi=True)
    assert np.abs(kt - okt[0, 0]).max() > 1e-3 * np.abs(kt).max()
