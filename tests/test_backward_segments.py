"""The segment-parallel form of the Phase 1 adjoint, checked in fp64 against
the sequential adjoint (``test_backward_algebra.phase1_adjoint``, itself
checked against the autograd reference gradients).

The adjoint of the preconditioner scan ("OSDN: Improving Delta Rule with
Provable Online Preconditioning in Linear Attention", gist.science summary,
sections 2.2-2.3, differentiated) is linear in lam:
    lam_t = (r_t I - mu_t w_t w_t^T) lam_{t+1} + g_t,   mu_t = eta beta_t^2 / n_t,
so, as the forward scan does for d, a sequence splits into time segments
run in parallel: segment [s, e) starts lam from zero W tokens past e (the
last segment from the exact d_dT at T), walks back to s, and is verified
from the last segment to the first: where its speculative lam at e differs
from the exact lam the next segment produced at its start by more than
2^-21 relative, it is walked again from that exact value.  The per-token
outputs of a segment are those of its (final) walk.  The exact d at every
segment start comes from the forward scan.

With a retention gate the warm-up forgets its start and no segment is
repaired; with slow retention (r near 1) segments are repaired and the
result is still exact -- both are checked.
"""
import numpy as np
import pytest

from tests.test_backward_algebra import phase1_adjoint

REL_TOL = 2.0 ** -21


def forward_d(k, beta, r, eta, d0):
    T, K = k.shape
    d = d0.copy()
    ds = np.zeros((T + 1, K))
    for t in range(T):
        ds[t] = d
        w = k[t] ** 2
        n = w.sum()
        c = eta * beta[t] * (1 - beta[t] * (d @ w)) / n if n > 0 else 0.0
        d = r[t] * d + c * w
    ds[T] = d
    return ds


def walk(lam, t_hi, t_lo, k, beta, r, eta, ds, g, dk2, db2, out):
    """lam at t_hi -> lam at t_lo; writes per-token outputs into `out` when given."""
    for t in range(t_hi - 1, t_lo - 1, -1):
        d, kk, bt = ds[t], k[t], beta[t]
        w = kk ** 2
        n = w.sum()
        a = d @ w
        dc = lam @ w
        if n > 0:
            c = eta * bt * (1 - bt * a) / n
            da = -dc * eta * bt * bt / n
            db1 = dc * eta * (1 - 2 * bt * a) / n
            de = dc * bt * (1 - bt * a) / n
            dn = -dc * c / n
        else:
            c = da = db1 = de = dn = 0.0
        if out is not None:
            out["dr"][t] = lam @ d
            out["dk"][t] = dk2[t] + g[t] * d + 2 * kk * (c * lam + da * d + dn)
            out["dbeta"][t] = db2[t] + db1
            out["deta"][t] = de
        lam = r[t] * lam + da * w + g[t] * kk
    return lam


def segmented_adjoint(k, beta, r, eta, d0, g, ddT, dk2, db2, L, W=128):
    T, K = k.shape
    ds = forward_d(k, beta, r, eta, d0)      # the scan's exact segment starts (and every d_t)
    nseg = -(-T // L)
    out = {"dr": np.zeros(T), "dk": np.zeros((T, K)), "dbeta": np.zeros(T), "deta": np.zeros(T)}
    spec_end, start = [None] * nseg, [None] * nseg
    for i in range(nseg):                    # in parallel on the GPU
        s, e = i * L, min(T, (i + 1) * L)
        if e == T:
            lam = ddT.copy()
        else:
            lam = walk(np.zeros(K), min(T, e + W), e, k, beta, r, eta, ds, g, dk2, db2, None)
            if min(T, e + W) == T:           # the warm-up reached T: start it exactly
                lam = walk(ddT.copy(), T, e, k, beta, r, eta, ds, g, dk2, db2, None)
        spec_end[i] = lam
        start[i] = walk(lam, e, s, k, beta, r, eta, ds, g, dk2, db2, out)
    repaired = 0
    for i in range(nseg - 2, -1, -1):        # verify, last segment first
        exact = start[i + 1]
        diff = np.abs(spec_end[i] - exact).max()
        if not diff <= REL_TOL * np.abs(exact).max():
            s, e = i * L, min(T, (i + 1) * L)
            start[i] = walk(exact.copy(), e, s, k, beta, r, eta, ds, g, dk2, db2, out)
            repaired += 1
    return dict(dk=out["dk"], dbeta=out["dbeta"], dr=out["dr"], dd0=start[0],
                deta=out["deta"].sum()), repaired


def inputs(T, K, seed, slow):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((T, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    beta = 1 / (1 + np.exp(-rng.standard_normal(T)))
    r = 1 - 1e-4 * rng.random(T) if slow else 1 / (1 + np.exp(-(rng.standard_normal(T) + 2)))
    d0 = 0.5 + rng.random(K)
    g = rng.standard_normal((T, K))
    ddT = rng.standard_normal(K)
    dk2 = rng.standard_normal((T, K))
    db2 = rng.standard_normal(T)
    return k, beta, r, 0.1, d0, g, ddT, dk2, db2


def sequential(k, beta, r, eta, d0, g, ddT, dk2, db2):
    B = lambda x: x[None, None]
    res = phase1_adjoint(B(k), B(beta), B(r), eta, B(d0), B(g), B(ddT), B(dk2), B(db2))
    return {n: (v[0, 0] if n != "deta" else v) for n, v in res.items()}


@pytest.mark.parametrize("T,L,slow", [(1200, 256, False), (1000, 300, False), (900, 256, True)])
def test_segmented_adjoint_equals_sequential(T, L, slow):
    args = inputs(T, 16, 40 + T, slow)
    ref = sequential(*args)
    got, repaired = segmented_adjoint(*args, L=L)
    if slow:
        assert repaired > 0            # the repair path ran
    else:
        assert repaired == 0           # the warm-up alone was enough
    for n in ref:
        err = np.abs(np.asarray(got[n]) - ref[n]).max() / max(1e-300, np.abs(ref[n]).max())
        assert err < 1e-9, (n, err)
