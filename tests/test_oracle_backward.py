"""Pins for the fp64 reference gradients (``oracle.backward``), the oracle of
the backward pass that training through both phases needs.

(1) Its forward, a token-by-token float64 torch restatement, equals the C
    oracle's forward (``oracle.forward``) on every output.
(2) Its gradients equal central finite differences of the C oracle's
    forward, element by element, for every input including eta: the
    difference quotients use nothing of autograd or of the torch forward.
"""
import numpy as np
import pytest

import oracle
from oracle import backward
from preconditioned_delta_rule_phase1_gb300 import synth


def case(gated, seed, T=6, K=4, V=3):
    x = synth.make_random(1, 2, T, K, V, io="f32", apf=True, gated=gated, s0=True, d0=True,
                          seed=seed)
    return {n: (t.double().numpy() if hasattr(t, "numpy") else t) for n, t in x.items()}


@pytest.mark.parametrize("gated", [False, True])
def test_torch_forward_equals_c_oracle(gated):
    x = case(gated, 61, T=23, K=8, V=5)
    ref = oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"],
                         x["alpha"], x["S0"])
    t = {n: backward._t(x[n]) for n in ("q", "k", "v", "beta", "r", "d0", "alpha", "S0")}
    got = backward.forward_torch(t["q"], t["k"], t["v"], t["beta"], t["r"], x["eta"], t["d0"],
                                 t["alpha"], t["S0"])
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g.numpy(), r, rtol=0, atol=1e-12 * max(1.0, np.abs(r).max()))


def c_loss(x, cot):
    kt, dT, o, ST = oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"],
                                   x["alpha"], x["S0"], nthreads=1)
    return (np.sum(o * cot["o"]) + np.sum(dT * cot["dT"]) + np.sum(ST * cot["ST"])
            + np.sum(kt * cot["kt"]))


@pytest.mark.parametrize("gated", [False, True])
def test_gradients_equal_finite_differences(gated):
    x = case(gated, 62)
    rng = np.random.default_rng(5)
    kt, dT, o, ST = oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"],
                                   x["alpha"], x["S0"])
    cot = {"o": rng.standard_normal(o.shape), "dT": rng.standard_normal(dT.shape),
           "ST": rng.standard_normal(ST.shape), "kt": rng.standard_normal(kt.shape)}
    g = backward.grads(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"], x["alpha"],
                       x["S0"], do=cot["o"], ddT=cot["dT"], dST=cot["ST"], dkt=cot["kt"])
    h = 1e-6
    names = ["q", "k", "v", "beta", "r", "d0", "S0", "eta"] + (["alpha"] if gated else [])
    for n in names:
        if n == "eta":
            xp, xm = dict(x), dict(x)
            xp["eta"], xm["eta"] = x["eta"] + h, x["eta"] - h
            fd = (c_loss(xp, cot) - c_loss(xm, cot)) / (2 * h)
            assert abs(g["eta"] - fd) <= 1e-6 * max(1.0, abs(fd)), (n, g["eta"], fd)
            continue
        base = x[n]
        num = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            xp, xm = dict(x), dict(x)
            xp[n], xm[n] = base.copy(), base.copy()
            xp[n][idx] += h
            xm[n][idx] -= h
            num[idx] = (c_loss(xp, cot) - c_loss(xm, cot)) / (2 * h)
        scale = max(1.0, np.abs(num).max())
        np.testing.assert_allclose(g[n], num, rtol=0, atol=1e-6 * scale, err_msg=n)


def test_finite_differences_catch_a_dropped_retention_gate():
    # the gradient of a forward with r left out must not pass the comparison
    # above: it is sensitive to the retention gate's terms
    x = case(False, 63)
    rng = np.random.default_rng(6)
    kt, dT, o, ST = oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"],
                                   x["alpha"], x["S0"])
    cot = {"o": rng.standard_normal(o.shape), "dT": rng.standard_normal(dT.shape),
           "ST": rng.standard_normal(ST.shape), "kt": rng.standard_normal(kt.shape)}
    wrong = backward.grads(x["q"], x["k"], x["v"], x["beta"], None, x["eta"], x["d0"], None,
                           x["S0"], do=cot["o"], ddT=cot["dT"], dST=cot["ST"], dkt=cot["kt"])
    h = 1e-6
    base = x["d0"]
    num = np.zeros_like(base)
    for idx in np.ndindex(base.shape):
        xp, xm = dict(x), dict(x)
        xp["d0"], xm["d0"] = base.copy(), base.copy()
        xp["d0"][idx] += h
        xm["d0"][idx] -= h
        num[idx] = (c_loss(xp, cot) - c_loss(xm, cot)) / (2 * h)
    assert np.abs(wrong["d0"] - num).max() > 1e-3 * max(1.0, np.abs(num).max())


def test_stored_ktilde_option():
    # (1) with the exact ktilde the straight-through value changes nothing;
    # (2) with a perturbed ktilde the forward is the C oracle's Phase 2 on
    #     that ktilde (a separate implementation of the recurrence)
    x = case(True, 64)
    kt, dT, o, ST = oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"],
                                   x["alpha"], x["S0"])
    rng = np.random.default_rng(9)
    cot = {"do": rng.standard_normal(o.shape), "dST": rng.standard_normal(ST.shape)}
    plain = backward.grads(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"],
                           x["alpha"], x["S0"], **cot)
    same = backward.grads(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"],
                          x["alpha"], x["S0"], ktilde=kt, **cot)
    for n in plain:
        np.testing.assert_allclose(same[n], plain[n], rtol=0,
                                   atol=1e-12 * max(1.0, np.abs(plain[n]).max()), err_msg=n)
    kt2 = kt * (1 + 1e-2 * rng.standard_normal(kt.shape))
    t = {n: backward._t(x[n]) for n in ("q", "k", "v", "beta", "r", "d0", "alpha", "S0")}
    _, _, o2, S2 = backward.forward_torch(t["q"], t["k"], t["v"], t["beta"], t["r"], x["eta"],
                                          t["d0"], t["alpha"], t["S0"], backward._t(kt2))
    o_ref, S_ref = oracle.delta_fwd(x["q"], x["k"], kt2, x["v"], x["beta"], x["alpha"], x["S0"])
    np.testing.assert_allclose(o2.numpy(), o_ref, rtol=0, atol=1e-12 * np.abs(o_ref).max())
    np.testing.assert_allclose(S2.numpy(), S_ref, rtol=0, atol=1e-12 * np.abs(S_ref).max())
