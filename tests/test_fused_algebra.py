"""The rebuild of the preconditioned keys that the fused forward pass runs
on the tensor cores, checked in fp64 against the oracle's scan.

Inside a chunk of 64 tokens that starts from d_c, the preconditioner step
d_{t+1} = r_t d_t + e_t w_t (w = k . k; gist.science summary of arXiv
2605.13473, sections 2.2-2.3) unrolls to

    d_t = rho_t d_c + sum_{u<t} pi_ut e_u w_u,
    rho_t = prod_{v<t} r_v,   pi_ut = prod_{u<v<t} r_v,

i.e. D = rho d_c^T + P W with P_tu = pi_ut e_u (u < t).  The fused pass
stores e_t and d_c instead of ktilde and evaluates this product per chunk.
Here e_t and d_t are read off the oracle's own scan (d_t = ktilde_t / k_t,
e_t from d_{t+1} - r_t d_t along w_t), and the chunk formula must give back
every d_t.  An index slip in pi (the factor r_t of the token itself
included) fails.
"""
import numpy as np
import pytest

import oracle
from preconditioned_delta_rule_phase1_gb300 import synth


def scan_states(x, h):
    """d_t for t = 0..T (d_T last) and e_t of sequence h, from the oracle."""
    kt, dT = oracle.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"])
    k = x["k"][0, h].double().numpy()
    d = np.asarray(kt)[0, h] / k                        # d_t = ktilde_t / k_t (keys are nonzero)
    d = np.vstack([d, np.asarray(dT)[0, h][None]])       # append d_T
    r = np.ones(k.shape[0]) if x["r"] is None else x["r"][0, h].double().numpy()
    w = k * k
    step = d[1:] - r[:, None] * d[:-1]                   # = e_t w_t
    e = (step * w).sum(1) / (w * w).sum(1)
    return d, e, r, w


def rebuild(d_c, e, r, w, off_by_one=False):
    n = len(e)
    rho = np.concatenate([[1.0], np.cumprod(r[:-1])])   # prod_{v<t} r_v
    P = np.zeros((n, n))
    for t in range(n):
        for u in range(t):
            lo = u if off_by_one else u + 1
            P[t, u] = np.prod(r[lo:t]) * e[u]
    return rho[:, None] * d_c[None, :] + P @ w


@pytest.mark.parametrize("T,apf,h", [(300, True, 0), (300, False, 1), (130, True, 2), (64, True, 0)])
def test_chunk_rebuild_equals_the_scan(T, apf, h):
    x = synth.make_random(1, 3, T, 64, 64, io="f32", apf=apf, d0=True, eta=0.5, seed=T + h)
    d, e, r, w = scan_states(x, h)
    for c0 in range(0, T, 64):
        c1 = min(T, c0 + 64)
        D = rebuild(d[c0], e[c0:c1], r[c0:c1], w[c0:c1])
        np.testing.assert_allclose(D, d[c0:c1], rtol=0, atol=1e-12 * np.abs(d[c0:c1]).max())


def test_chunk_rebuild_catches_an_index_slip():
    x = synth.make_random(1, 1, 128, 64, 64, io="f32", apf=True, d0=True, eta=0.5, seed=7)
    d, e, r, w = scan_states(x, 0)
    D = rebuild(d[64], e[64:128], r[64:128], w[64:128], off_by_one=True)
    assert np.abs(D - d[64:128]).max() > 1e-4 * np.abs(d[64:128]).max()
