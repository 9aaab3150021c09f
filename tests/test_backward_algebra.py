"""The reverse-time recurrences of the GPU backward pass, checked in fp64 on
the CPU against the reference gradients (``oracle.backward``, fp64 autograd,
itself pinned by finite differences of the C oracle).

The kernels in ``csrc/backward.cu`` follow the derivative of the forward of
"OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear
Attention" (gist.science summary, sections 2.1-2.3) taken by hand, in the
decomposition written out below:

Phase 2, one value row i of S at a time (rows evolve independently), state
checkpoints every SUB tokens, each sub-chunk recomputed forward and then
walked backwards with the row's state gradient G = dL/dS_t[i, :]:

    G += dO_t[i] q_t                       (o_t = S_t q_t)
    du = <G, ktilde_t>                     (S_t = S_bar + u ktilde^T)
    dS_bar = G - beta_t du k_t             (u = beta (v - S_bar k))
    row contributions, summed over rows in fixed row-block order:
        dq_t     += dO_t[i] S_t[i]
        dktilde_t += u_t[i] G
        dk_t     += -beta_t du alpha_t S_{t-1}[i]
        dbeta_t  += du e_t[i],  e = v - S_bar k
        dalpha_t += <dS_bar, S_{t-1}[i]>
    dv_t[i] = beta_t du;  G = alpha_t dS_bar;  dS0[i] = G at the start.

Phase 1, one sequence at a time, the adjoint lam = dL/dd_t run backwards
(its step is the transpose of the forward's linear part, which is symmetric):

    dr_t = <lam, d_t>,  dc = <lam, w_t>,  c_t = eta beta (1 - beta a)/n
    da = -dc eta beta^2 / n,  dbeta += dc eta (1 - 2 beta a)/n,
    deta += dc beta (1 - beta a)/n,  dn = -dc c_t / n      (0 if n = 0)
    dk_t += g d_t + 2 k (c_t lam + da d_t + dn),  g = dktilde_t (both parts)
    lam = r_t lam + da w_t + g k_t;  dd0 = lam at the start.

A test below drops one term and checks that the comparison catches it.  The
last test runs the per-channel-decay variant (Diag(alpha_t) in place of
alpha_t, dalpha_t[j] += dS_bar[i, j] S_{t-1}[i, j]) as the kernels' PCH flag
does, against the autograd gradients with a [B, H, T, K] decay.
"""
import numpy as np
import pytest

from oracle import backward
from preconditioned_delta_rule_phase1_gb300 import synth

SUB = 16   # tokens per recomputed sub-chunk (both kernels)
RB = 8     # value rows per row block of the Phase 2 kernel


def phase2_adjoint(q, k, kt, v, beta, alpha, S0, dO, dST, drop=None):
    B, H, T, K = k.shape
    V = v.shape[-1]
    P = 3 * K + 2
    part = np.zeros((B, H, V // RB, T, P))
    dv = np.zeros((B, H, T, V))
    dS0 = np.zeros((B, H, V, K))
    for b in range(B):
        for h in range(H):
            for i in range(V):
                rb = i // RB
                S = S0[b, h, i].copy()
                ck = []
                for t in range(T):
                    if t % SUB == 0:
                        ck.append(S.copy())
                    a = alpha[b, h, t]
                    u = beta[b, h, t] * (v[b, h, t, i] - a * (S @ k[b, h, t]))
                    S = a * S + u * kt[b, h, t]
                G = dST[b, h, i].copy()
                for j in reversed(range(len(ck))):
                    t0 = j * SUB
                    tn = min(SUB, T - t0)
                    Sp, us, es = [], [], []
                    S = ck[j].copy()
                    for tt in range(tn):
                        t = t0 + tt
                        a = alpha[b, h, t]
                        e = v[b, h, t, i] - a * (S @ k[b, h, t])
                        u = beta[b, h, t] * e
                        Sp.append(S.copy())
                        es.append(e)
                        us.append(u)
                        S = a * S + u * kt[b, h, t]
                    for tt in reversed(range(tn)):
                        t = t0 + tt
                        a, bt = alpha[b, h, t], beta[b, h, t]
                        St = a * Sp[tt] + us[tt] * kt[b, h, t]
                        if drop != "readout":
                            G = G + dO[b, h, t, i] * q[b, h, t]
                        du = G @ kt[b, h, t]
                        dSb = G - bt * du * k[b, h, t]
                        pr = part[b, h, rb, t]
                        pr[0:K] += dO[b, h, t, i] * St
                        pr[K:2 * K] += us[tt] * G
                        pr[2 * K:3 * K] += -bt * du * a * Sp[tt]
                        pr[3 * K] += du * es[tt]
                        pr[3 * K + 1] += dSb @ Sp[tt]
                        dv[b, h, t, i] = bt * du
                        G = a * dSb
                dS0[b, h, i] = G
    tot = np.zeros((B, H, T, P))
    for rb in range(V // RB):          # fixed order, as the reduce kernel sums
        tot += part[:, :, rb]
    return dict(dq=tot[..., 0:K], dkt=tot[..., K:2 * K], dk2=tot[..., 2 * K:3 * K],
                dbeta2=tot[..., 3 * K], dalpha=tot[..., 3 * K + 1], dv=dv, dS0=dS0)


def phase1_adjoint(k, beta, r, eta, d0, g_all, ddT, dk2, dbeta2, drop=None):
    B, H, T, K = k.shape
    dk = np.zeros_like(k)
    dbeta = np.zeros_like(beta)
    dr = np.zeros_like(beta)
    dd0 = np.zeros((B, H, K))
    deta = np.zeros((B, H))
    for b in range(B):
        for h in range(H):
            d = d0[b, h].copy()
            ck = []
            for t in range(T):
                if t % SUB == 0:
                    ck.append(d.copy())
                w = k[b, h, t] ** 2
                n = w.sum()
                c = eta * beta[b, h, t] * (1 - beta[b, h, t] * (d @ w)) / n if n > 0 else 0.0
                d = r[b, h, t] * d + c * w
            lam = ddT[b, h].copy()
            for j in reversed(range(len(ck))):
                t0 = j * SUB
                tn = min(SUB, T - t0)
                ds = []
                d = ck[j].copy()
                for tt in range(tn):
                    t = t0 + tt
                    w = k[b, h, t] ** 2
                    n = w.sum()
                    c = eta * beta[b, h, t] * (1 - beta[b, h, t] * (d @ w)) / n if n > 0 else 0.0
                    ds.append(d.copy())
                    d = r[b, h, t] * d + c * w
                for tt in reversed(range(tn)):
                    t = t0 + tt
                    d, kk, bt = ds[tt], k[b, h, t], beta[b, h, t]
                    w = kk ** 2
                    n = w.sum()
                    a = d @ w
                    dr[b, h, t] = lam @ d
                    dc = lam @ w
                    if n > 0:
                        c = eta * bt * (1 - bt * a) / n
                        da = -dc * eta * bt * bt / n
                        db1 = dc * eta * (1 - 2 * bt * a) / n
                        deta[b, h] += dc * bt * (1 - bt * a) / n
                        dn = -dc * c / n
                    else:
                        c = da = db1 = dn = 0.0
                    if drop == "da":
                        da = 0.0
                    g = g_all[b, h, t]
                    dk[b, h, t] = dk2[b, h, t] + g * d + 2 * kk * (c * lam + da * d + dn)
                    dbeta[b, h, t] = dbeta2[b, h, t] + db1
                    lam = r[b, h, t] * lam + da * w + g * kk
            dd0[b, h] = lam
    return dict(dk=dk, dbeta=dbeta, dr=dr, dd0=dd0, deta=deta.sum())


def by_hand(x, cot, drop=None):
    B, H, T, K = x["k"].shape
    V = x["v"].shape[-1]
    ones = np.ones((B, H, T))
    r = x["r"] if x["r"] is not None else ones
    alpha = x["alpha"] if x["alpha"] is not None else ones
    d0 = x["d0"] if x["d0"] is not None else np.ones((B, H, K))
    S0 = x["S0"] if x["S0"] is not None else np.zeros((B, H, V, K))
    # ktilde as the forward makes it (d_t before the step, times k_t)
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
    p2 = phase2_adjoint(x["q"], x["k"], kt, x["v"], x["beta"], alpha, S0, cot["o"], cot["ST"],
                        drop)
    g_all = p2["dkt"] + cot["kt"]
    p1 = phase1_adjoint(x["k"], x["beta"], r, x["eta"], d0, g_all, cot["dT"], p2["dk2"],
                        p2["dbeta2"], drop)
    return dict(q=p2["dq"], k=p1["dk"], v=p2["dv"], beta=p1["dbeta"], r=p1["dr"],
                alpha=p2["dalpha"], d0=p1["dd0"], S0=p2["dS0"], eta=p1["deta"])


def case(T, K, V, seed, gated=True, zero_key=False):
    x = synth.make_random(1, 2, T, K, V, io="f32", apf=True, gated=gated, s0=True, d0=True,
                          seed=seed)
    x = {n: (t.double().numpy() if hasattr(t, "numpy") else t) for n, t in x.items()}
    if zero_key:
        x["k"][0, 1, 3] = 0.0
    rng = np.random.default_rng(seed + 100)
    B, H = 1, 2
    cot = {"o": rng.standard_normal((B, H, T, V)), "dT": rng.standard_normal((B, H, K)),
           "ST": rng.standard_normal((B, H, V, K)), "kt": rng.standard_normal((B, H, T, K))}
    return x, cot


def reference(x, cot):
    return backward.grads(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"],
                          x["alpha"], x["S0"], do=cot["o"], ddT=cot["dT"], dST=cot["ST"],
                          dkt=cot["kt"])


def worst(got, ref, names):
    err = {}
    for n in names:
        g, r = np.asarray(got[n], float), np.asarray(ref[n], float)
        err[n] = float(np.abs(g - r).max() / max(1e-30, np.abs(r).max()))
    return err


NAMES = ["q", "k", "v", "beta", "r", "alpha", "d0", "S0", "eta"]


@pytest.mark.parametrize("T,K,V,gated,zero_key", [
    (37, 8, 16, True, False),      # two full sub-chunks and a ragged tail
    (16, 4, 8, False, False),      # exactly one sub-chunk, ungated
    (5, 8, 8, True, True),         # shorter than a sub-chunk, a zero key
    (48, 6, 24, True, False),      # three sub-chunks, three row blocks
])
def test_recurrences_match_reference_gradients(T, K, V, gated, zero_key):
    x, cot = case(T, K, V, 70 + T, gated, zero_key)
    ref = reference(x, cot)
    got = by_hand(x, cot)
    names = [n for n in NAMES if n in ref]
    err = worst(got, ref, names)
    assert max(err.values()) < 1e-11, err


@pytest.mark.parametrize("drop", ["readout", "da"])
def test_a_dropped_term_is_caught(drop):
    x, cot = case(21, 8, 8, 91)
    ref = reference(x, cot)
    err = worst(by_hand(x, cot, drop), ref, NAMES)
    assert max(err.values()) > 1e-3, err


def phase2_adjoint_per_channel(q, k, kt, v, beta, alpha_k, S0, dO, dST):
    """The state adjoint with a decay per key channel, as the kernel's PCH
    variant runs it: Diag(alpha_t) in place of alpha_t, dalpha_t per column."""
    B, H, T, K = k.shape
    V = v.shape[-1]
    dq, dkt, dk2 = np.zeros_like(q), np.zeros_like(k), np.zeros_like(k)
    db2, da = np.zeros((B, H, T)), np.zeros((B, H, T, K))
    dv, dS0 = np.zeros_like(v), np.zeros((B, H, V, K))
    for b in range(B):
        for h in range(H):
            for i in range(V):
                S = S0[b, h, i].copy()
                Sp, es, us = [], [], []
                for t in range(T):
                    a = alpha_k[b, h, t]
                    e = v[b, h, t, i] - (a * S) @ k[b, h, t]
                    u = beta[b, h, t] * e
                    Sp.append(S.copy())
                    es.append(e)
                    us.append(u)
                    S = a * S + u * kt[b, h, t]
                G = dST[b, h, i].copy()
                for t in reversed(range(T)):
                    a, bt = alpha_k[b, h, t], beta[b, h, t]
                    St = a * Sp[t] + us[t] * kt[b, h, t]
                    G = G + dO[b, h, t, i] * q[b, h, t]
                    du = G @ kt[b, h, t]
                    dSb = G - bt * du * k[b, h, t]
                    dq[b, h, t] += dO[b, h, t, i] * St
                    dkt[b, h, t] += us[t] * G
                    dk2[b, h, t] += -bt * du * a * Sp[t]
                    db2[b, h, t] += du * es[t]
                    da[b, h, t] += dSb * Sp[t]
                    dv[b, h, t, i] = bt * du
                    G = a * dSb
                dS0[b, h, i] = G
    return dict(dq=dq, dkt=dkt, dk2=dk2, dbeta2=db2, dalpha=da, dv=dv, dS0=dS0)


def test_per_channel_decay_recurrences_match_reference():
    x, cot = case(23, 8, 8, 121, gated=False)
    rng = np.random.default_rng(122)
    B, H, T, K = x["k"].shape
    x["alpha"] = 0.6 + 0.4 * rng.random((B, H, T, K))
    ref = reference(x, cot)
    d0 = x["d0"]
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
                d = x["r"][b, h, t] * d + c * w
    p2 = phase2_adjoint_per_channel(x["q"], x["k"], kt, x["v"], x["beta"], x["alpha"], x["S0"],
                                    cot["o"], cot["ST"])
    p1 = phase1_adjoint(x["k"], x["beta"], x["r"], x["eta"], d0, p2["dkt"] + cot["kt"],
                        cot["dT"], p2["dk2"], p2["dbeta2"])
    got = dict(q=p2["dq"], k=p1["dk"], v=p2["dv"], beta=p1["dbeta"], r=p1["dr"],
               alpha=p2["dalpha"], d0=p1["dd0"], S0=p2["dS0"], eta=p1["deta"])
    err = worst(got, ref, list(ref))
    assert max(err.values()) < 1e-11, err
