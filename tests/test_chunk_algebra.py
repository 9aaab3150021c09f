"""The chunk algebra the tensor-core kernels evaluate, checked in fp64.

The Phase 2 kernels do not run the token recurrence of the gist.science
summary of arXiv 2605.13473 (section 2.1) directly: per chunk of 64 tokens
they form, from the keys alone,

    L  = tril(diag(b) (G . K Kt^T), -1),   A  = tril(G . Q Kt^T),
    X  = (I + L)^-1,  Xb = X diag(b),      Kw = Xb diag(g) K,
    W  = (D Kt)^T Xb,  M = -(D Kt)^T Kw,   Ae = A Xb,  Qe = diag(g) Q - A Kw,

(g the within-chunk cumulative product of alpha, G_ij = g_i / g_j,
D = diag(g_C / g)) and then carry the state with one product per chunk:

    O = Ae V + Qe S^T,    S'^T = g_C S^T + W V + M S^T.

This test restates that algebra in plain fp64 numpy, chunk by chunk, and
compares it with the fp64 oracle's token recurrence.  It pins the
derivation the kernels rely on (a wrong sign, a transposed operand or a
misplaced decay in it fails here), independently of any GPU code.
"""
import numpy as np
import pytest

import oracle
from preconditioned_delta_rule_phase1_gb300 import synth


def chunk_form(q, k, kt, v, beta, alpha, S0, C=64):
    """Phase 2 for one sequence by the per-chunk algebra above (fp64)."""
    T, K = k.shape
    V = v.shape[1]
    S = np.zeros((V, K)) if S0 is None else S0.astype(np.float64).copy()
    o = np.zeros((T, V))
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        Q, Kc, Kt, Vc, b = q[c0:c0 + n], k[c0:c0 + n], kt[c0:c0 + n], v[c0:c0 + n], beta[c0:c0 + n]
        lg = np.cumsum(np.log(alpha[c0:c0 + n])) if alpha is not None else np.zeros(n)
        g = np.exp(lg)
        G = np.exp(lg[:, None] - lg[None, :])
        L = np.tril(b[:, None] * G * (Kc @ Kt.T), -1)
        A = np.tril(G * (Q @ Kt.T))
        X = np.linalg.inv(np.eye(n) + L)
        Xb = X * b[None, :]
        Kw = Xb @ (g[:, None] * Kc)
        Dkt = (g[-1] / g)[:, None] * Kt
        W = Dkt.T @ Xb
        M = -Dkt.T @ Kw
        Ae = A @ Xb
        Qe = g[:, None] * Q - A @ Kw
        o[c0:c0 + n] = Ae @ Vc + Qe @ S.T
        S = (g[-1] * S.T + W @ Vc + M @ S.T).T
    return o, S


@pytest.mark.parametrize("T,gated,s0", [(64, False, False), (200, True, True), (257, False, True),
                                        (130, True, False)])
def test_chunk_algebra_equals_token_recurrence(T, gated, s0):
    x = synth.make_random(1, 2, T, 32, 16, io="f32", apf=True, gated=gated, s0=s0, seed=T)
    f64 = lambda t: None if t is None else t.double().numpy()
    kt, _ = oracle.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"])
    o_ref, S_ref = oracle.delta_fwd(x["q"], x["k"], kt, x["v"], x["beta"], x["alpha"], x["S0"])
    q, k, v, beta = f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["beta"])
    alpha, S0 = f64(x["alpha"]), f64(x["S0"])
    kt = np.asarray(kt, dtype=np.float64)
    for h in range(2):
        o, S = chunk_form(q[0, h], k[0, h], kt[0, h], v[0, h], beta[0, h],
                          None if alpha is None else alpha[0, h], None if S0 is None else S0[0, h])
        np.testing.assert_allclose(o, np.asarray(o_ref)[0, h], rtol=0, atol=1e-10 * np.abs(o).max())
        np.testing.assert_allclose(S, np.asarray(S_ref)[0, h], rtol=0, atol=1e-10 * np.abs(S).max())


def test_chunk_algebra_catches_a_dropped_decay():
    # the same algebra with the state decay g_C left out must not pass: the
    # comparison above is sensitive to the terms that carry the gate
    x = synth.make_random(1, 1, 130, 32, 16, io="f32", apf=True, gated=True, s0=True, seed=5)
    f64 = lambda t: None if t is None else t.double().numpy()
    kt, _ = oracle.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"])
    o_ref, _ = oracle.delta_fwd(x["q"], x["k"], kt, x["v"], x["beta"], x["alpha"], x["S0"])
    kt = np.asarray(kt, dtype=np.float64)
    o, _ = chunk_form(f64(x["q"])[0, 0], f64(x["k"])[0, 0], kt[0, 0], f64(x["v"])[0, 0],
                      f64(x["beta"])[0, 0], np.ones(130), f64(x["S0"])[0, 0])
    assert np.abs(o - np.asarray(o_ref)[0, 0]).max() > 1e-3 * np.abs(o).max()
