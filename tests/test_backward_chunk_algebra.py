"""The chunked form of Phase 2's backward, checked in fp64 against the
reference gradients (``oracle.backward``: autograd through the token
recurrence, pinned by finite differences of the C oracle).

This is the algebra a tensor-core backward evaluates: per chunk of C tokens
the forward of the tensor-core kernels (gist.science summary of "OSDN:
Improving Delta Rule with Provable Online Preconditioning in Linear
Attention", section 2.1: the chunkwise pipeline with Ktilde in the Gram
matrix and the scores), with Sigma = S^T (K x V) at the chunk start,

    G_ij = g_i / g_j,  g the within-chunk cumulative product of alpha
    P = G . K Kt^T,    L = tril(diag(b) P, -1),   A = tril(G . Q Kt^T)
    X = (I + L)^-1,    Xb = X diag(b)
    R = V - diag(g) K Sigma,   U = Xb R
    O = A U + diag(g) Q Sigma,   Sigma' = g_C Sigma + (diag(g_C / g) Kt)^T U

differentiated by hand, chunk by chunk in reverse with the state gradient
dSigma carried between chunks:

    dU = A^T dO + diag(g_C/g) Kt dSigma'
    dSigma = g_C dSigma' + (diag(g) Q)^T dO - (diag(g) K)^T Xb^T dU
    dV = Xb^T dU,   dA = tril(dO U^T),   dXb = dU R^T
    dL = -tril(X^T (dXb diag(b)) X^T, -1)
    dQ = diag(g) dO Sigma^T + (G . dA) Kt
    dK = -diag(g) Xb^T dU Sigma^T + (G . diag(b) dL) Kt
    dKt = diag(g_C/g) U dSigma'^T + (G . diag(b) dL)^T K + (G . dA)^T Q
    db = colsum(X . dXb) + rowsum(dL . P)
    and dalpha through log g: the gradient of G, g, g_C and g_C/g with
    respect to log g, then a reverse cumulative sum, divided by alpha.

The Phase 1 adjoint then takes dKt (``test_backward_algebra.phase1_adjoint``)
and the sum must equal the reference for every input.  A dropped decay term
fails the comparison.  A last test shows that the serial part, dSigma and
dV, needs only the forward's prepared operands transposed.
"""
import numpy as np
import pytest

from tests.test_backward_algebra import case, phase1_adjoint, reference, worst


def chunk_backward(q, k, kt, v, beta, alpha, S0, dO, dST, C=64, drop=None):
    """Phase 2's gradients for one sequence by the chunk algebra above."""
    T, K = k.shape
    a = np.ones(T) if alpha is None else alpha
    Sig = [S0.T.copy()]
    saved = []
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        sl = slice(c0, c0 + n)
        Q, Kc, Kt, Vc, b = q[sl], k[sl], kt[sl], v[sl], beta[sl]
        lg = np.cumsum(np.log(a[sl]))
        g = np.exp(lg)
        G = np.exp(lg[:, None] - lg[None, :])
        KK = Kc @ Kt.T
        QK = Q @ Kt.T
        P = G * KK
        L = np.tril(b[:, None] * P, -1)
        A = np.tril(G * QK)
        X = np.linalg.inv(np.eye(n) + L)
        Xb = X * b[None, :]
        Sg = Sig[-1]
        R = Vc - g[:, None] * (Kc @ Sg)
        U = Xb @ R
        gC = g[-1]
        dec = gC / g
        Sig.append(gC * Sg + (dec[:, None] * Kt).T @ U)
        saved.append(dict(sl=sl, Q=Q, Kc=Kc, Kt=Kt, b=b, g=g, G=G, KK=KK, QK=QK, P=P, A=A, X=X,
                          Xb=Xb, R=R, U=U, gC=gC, dec=dec))
    dq, dk, dkt, dv = (np.zeros_like(q), np.zeros_like(k), np.zeros_like(kt), np.zeros_like(v))
    db_all, da_all = np.zeros(T), np.zeros(T)
    dSig = dST.T.copy()
    for ci in reversed(range(len(saved))):
        c = saved[ci]
        sl, Sg = c["sl"], Sig[ci]
        dOc = dO[sl]
        Q, Kc, Kt, b, g, G = c["Q"], c["Kc"], c["Kt"], c["b"], c["g"], c["G"]
        X, Xb, R, U, gC, dec = c["X"], c["Xb"], c["R"], c["U"], c["gC"], c["dec"]
        dU = c["A"].T @ dOc + (dec[:, None] * Kt) @ dSig
        dSg = gC * dSig + (g[:, None] * Q).T @ dOc
        dv[sl] = Xb.T @ dU
        dA = np.tril(dOc @ U.T)
        dgQ = dOc @ Sg.T
        dQ = g[:, None] * dgQ
        dg = (Q * dgQ).sum(1)
        dDkt = U @ dSig.T
        dKt = dec[:, None] * dDkt
        ddec = (Kt * dDkt).sum(1)
        dgC = (dSig * Sg).sum()
        dXb = dU @ R.T
        dR = Xb.T @ dU
        dSg -= (g[:, None] * Kc).T @ dR
        dgK = -dR @ Sg.T
        dKc = g[:, None] * dgK
        dg += (Kc * dgK).sum(1)
        dX = dXb * b[None, :]
        db = (X * dXb).sum(0)
        dL = np.tril(-X.T @ dX @ X.T, -1)
        db += (dL * c["P"]).sum(1)
        dP = b[:, None] * dL
        GdP = G * dP
        dKc += GdP @ Kt
        dKt += GdP.T @ Kc
        dG = dP * c["KK"]
        GdA = G * dA
        dQ += GdA @ Kt
        dKt += GdA.T @ Q
        dG += dA * c["QK"]
        GG = dG * G
        dlg = GG.sum(1) - GG.sum(0) + dg * g
        if drop != "decay":
            dlg[-1] += dgC * gC + (ddec * dec).sum()
            dlg -= ddec * dec
        da_all[sl] = np.cumsum(dlg[::-1])[::-1] / a[sl]
        dq[sl], dk[sl], dkt[sl], db_all[sl] = dQ, dKc, dKt, db
        dSig = dSg
    return dict(dq=dq, dk2=dk, dkt=dkt, dv=dv, dbeta2=db_all, dalpha=da_all, dS0=dSig.T)


def chunked(x, cot, C, drop=None):
    B, H, T, K = x["k"].shape
    V = x["v"].shape[-1]
    ones = np.ones((B, H, T))
    r = x["r"] if x["r"] is not None else ones
    d0 = x["d0"] if x["d0"] is not None else np.ones((B, H, K))
    S0 = x["S0"] if x["S0"] is not None else np.zeros((B, H, V, K))
    kt = np.zeros_like(x["k"])
    for b in range(B):
        for h in range(H):
            d = d0[b, h].copy()
            for t in range(T):
                kk = x["k"][b, h, t]
                kt[b, h, t] = d * kk
                w = kk ** 2
                n = w.sum()
                bt = x["beta"][b, h, t]
                c = x["eta"] * bt * (1 - bt * (d @ w)) / n if n > 0 else 0.0
                d = r[b, h, t] * d + c * w
    out = {n: np.zeros_like(v) for n, v in (("dq", x["q"]), ("dk2", x["k"]), ("dkt", x["k"]),
                                              ("dv", x["v"]), ("dbeta2", x["beta"]),
                                              ("dalpha", x["beta"]), ("dS0", S0))}
    for b in range(B):
        for h in range(H):
            res = chunk_backward(x["q"][b, h], x["k"][b, h], kt[b, h], x["v"][b, h],
                                 x["beta"][b, h], None if x["alpha"] is None else x["alpha"][b, h],
                                 S0[b, h], cot["o"][b, h], cot["ST"][b, h], C, drop)
            for n in out:
                out[n][b, h] = res[n]
    p1 = phase1_adjoint(x["k"], x["beta"], r, x["eta"], d0, out["dkt"] + cot["kt"], cot["dT"],
                        out["dk2"], out["dbeta2"])
    return dict(q=out["dq"], k=p1["dk"], v=out["dv"], beta=p1["dbeta"], r=p1["dr"],
                alpha=out["dalpha"], d0=p1["dd0"], S0=out["dS0"], eta=p1["deta"])


@pytest.mark.parametrize("T,K,V,gated,C", [
    (37, 8, 16, True, 16),      # two full chunks and a ragged tail
    (64, 6, 8, True, 64),       # one full chunk
    (50, 4, 8, False, 16),      # ungated
    (9, 8, 8, True, 64),        # shorter than a chunk
])
def test_chunked_backward_matches_reference(T, K, V, gated, C):
    x, cot = case(T, K, V, 170 + T, gated)
    ref = reference(x, cot)
    got = chunked(x, cot, C)
    names = [n for n in ref]
    err = worst(got, ref, names)
    assert max(err.values()) < 1e-10, err


def test_a_dropped_decay_term_is_caught():
    x, cot = case(40, 8, 8, 191, True)
    ref = reference(x, cot)
    err = worst(chunked(x, cot, 16, drop="decay"), ref, ["alpha"])
    assert err["alpha"] > 1e-3, err


def test_reverse_chain_is_the_forward_chain_transposed():
    # Per chunk the forward maps (V, Sigma) to (O, Sigma') linearly with the
    # prepared operands of the tensor-core forward,
    #     O = Ae V + Qe Sigma,   Sigma' = g_C Sigma + W V + M Sigma,
    # so the state gradient and dV need only those operands, transposed:
    #     dV = Ae^T dO + W^T dSigma',   dSigma = g_C dSigma' + M^T dSigma' + Qe^T dO.
    # Checked here against the explicit chunk backward above, chunk by chunk.
    x, cot = case(100, 8, 16, 211, True)
    h = 1
    q, k, v = x["q"][0, h], x["k"][0, h], x["v"][0, h]
    beta, alpha, S0 = x["beta"][0, h], x["alpha"][0, h], x["S0"][0, h]
    dO, dST = cot["o"][0, h], cot["ST"][0, h]
    rng = np.random.default_rng(5)
    kt = k * (0.5 + rng.random(k.shape))
    C, T = 32, 100
    ref = chunk_backward(q, k, kt, v, beta, alpha, S0, dO, dST, C)
    # forward with the prepared operands, keeping them per chunk
    ops_ = []
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        sl = slice(c0, c0 + n)
        Q, Kc, Kt, b = q[sl], k[sl], kt[sl], beta[sl]
        lg = np.cumsum(np.log(alpha[sl]))
        g = np.exp(lg)
        G = np.exp(lg[:, None] - lg[None, :])
        L = np.tril(b[:, None] * G * (Kc @ Kt.T), -1)
        A = np.tril(G * (Q @ Kt.T))
        Xb = np.linalg.inv(np.eye(n) + L) * b[None, :]
        Kw = Xb @ (g[:, None] * Kc)
        Dkt = (g[-1] / g)[:, None] * Kt
        ops_.append(dict(sl=sl, gC=g[-1], W=Dkt.T @ Xb, M=-Dkt.T @ Kw, Ae=A @ Xb,
                         Qe=g[:, None] * Q - A @ Kw))
    dSig = dST.T.copy()
    dv = np.zeros_like(v)
    for c in reversed(ops_):
        dOc = dO[c["sl"]]
        dv[c["sl"]] = c["Ae"].T @ dOc + c["W"].T @ dSig
        dSig = c["gC"] * dSig + c["M"].T @ dSig + c["Qe"].T @ dOc
    np.testing.assert_allclose(dv, ref["dv"], rtol=0, atol=1e-12 * np.abs(ref["dv"]).max())
    np.testing.assert_allclose(dSig.T, ref["dS0"], rtol=0, atol=1e-12 * np.abs(ref["dS0"]).max())
