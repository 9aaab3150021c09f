"""Pins for the fp64 oracle: each test checks the oracle against something
other than itself -- a special case the pages name, the definitional form of
the hypergradient surrogate, an identity of the quadratic inner loss, a dense
unrolled product, or a closed form of the preconditioner scan.

Sources (gist.science summary pages of "OSDN: Improving Delta Rule with
Provable Online Preconditioning in Linear Attention"):
  section 1    f_t(S) = 1/2||S k_t - v_t||^2; DeltaNet rule
  section 2.1  right-preconditioned update == preconditioned key ktilde = d.k
  section 2.2  definitional surrogate h_t and its closed form
  section 2.3  APF step on d with retention r
  section 3    theorem 5.2: residual ratios; gated Newton condition
"""
import fractions
import os

import numpy as np
import pytest

import oracle
from preconditioned_delta_rule_phase1_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(B=1, H=2, T=12, K=6, V=5, apf=False, gated=False, s0=False, seed=0):
    x = synth.make_random(B, H, T, K, V, io="f32", apf=apf, gated=gated, s0=s0, seed=seed)
    return {n: (t.double().numpy() if hasattr(t, "numpy") else t) for n, t in x.items()}


def f_loss(S, k, v):
    """f_t(S) = 1/2 ||S k - v||^2 (section 1)."""
    e = S @ k - v
    return 0.5 * float(e @ e)


def step_states(x, eta):
    """Run the oracle one token at a time, carrying (d, S); returns the
    per-token d_t (before the step), S_{t-1}, S_t for sequence (0, 0)."""
    T = x["k"].shape[2]
    d = None
    S = x["S0"][:, :1] if x["S0"] is not None else None
    out = []
    for t in range(T):
        sl = lambda a: None if a is None else a[:1, :1, t:t + 1]
        kt, dT = oracle.precond_scan(sl(x["k"]), sl(x["beta"]), sl(x["r"]), eta, d)
        o, ST = oracle.delta_fwd(sl(x["q"]), sl(x["k"]), kt, sl(x["v"]), sl(x["beta"]),
                                 sl(x["alpha"]), S)
        d_before = np.ones(x["k"].shape[-1]) if d is None else d[0, 0]
        S_before = np.zeros((x["v"].shape[-1], x["k"].shape[-1])) if S is None else S[0, 0]
        out.append((d_before, S_before, ST[0, 0], kt[0, 0, 0], o[0, 0, 0]))
        d, S = dT, ST
    return out


# ---------------------------------------------------------------------------
# (a) d = 1, eta = 0, r = 1 reduces to the DeltaNet rule (section 1 vs 2.1)
# ---------------------------------------------------------------------------
def test_pin_a_deltanet_special_case():
    x = rand_case(B=2, H=2, T=40, K=8, V=7, seed=1)
    kt, dT = oracle.precond_scan(x["k"], x["beta"], None, 0.0, None)
    assert np.array_equal(dT, np.ones_like(dT))
    assert np.array_equal(kt, x["k"])
    o, ST = oracle.delta_fwd(x["q"], x["k"], kt, x["v"], x["beta"])
    # textbook DeltaNet: S <- S + beta (v - S k) k^T, read-out S q
    for b in range(2):
        for h in range(2):
            S = np.zeros((7, 8))
            for t in range(40):
                k, v, q, be = x["k"][b, h, t], x["v"][b, h, t], x["q"][b, h, t], x["beta"][b, h, t]
                S = S + be * np.outer(v - S @ k, k)
                assert np.allclose(o[b, h, t], S @ q, rtol=0, atol=1e-14)
            assert np.allclose(ST[b, h], S, rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# (b) closed-form h_t equals the definitional surrogate computed from states
# (c) residual ratio f_t(S_t)/f_t(S_{t-1}) = (1 - beta <d, k^2>)^2
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("gated", [False, True])
def test_pin_b_c_surrogate_and_ratio(gated):
    x = rand_case(T=24, K=6, V=5, apf=True, gated=gated, s0=True, seed=2)
    eta = 0.3
    for t, (d, S_prev, S_new, kt, o) in enumerate(step_states(x, eta)):
        k, v, be = x["k"][0, 0, t], x["v"][0, 0, t], x["beta"][0, 0, t]
        al = x["alpha"][0, 0, t] if gated else 1.0
        Sb = al * S_prev                       # the state before the write
        n = float(k @ k)
        grad_f_sq = float(np.sum((Sb @ k - v) ** 2)) * n   # ||(S k - v) k^T||_F^2
        h_def = (f_loss(S_new, k, v) - f_loss(Sb, k, v)) / grad_f_sq
        a = float(d @ (k * k))
        h_closed = ((1.0 - be * a) ** 2 - 1.0) / (2.0 * n)
        assert abs(h_def - h_closed) <= 1e-10 * max(1.0, abs(h_closed)), t
        ratio = f_loss(S_new, k, v) / f_loss(Sb, k, v)
        assert abs(ratio - (1.0 - be * a) ** 2) <= 1e-10, t
        # the key written is d_t . k_t with the preconditioner before the step
        assert np.allclose(kt, d * k, rtol=0, atol=1e-15)
        # read-out from the state after the write
        assert np.allclose(o, S_new @ x["q"][0, 0, t], rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# q_geo: the log of the product of the residual ratios, from the states
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("gated", [False, True])
def test_pin_log_ratio_from_states(gated):
    """Phase 1's per-sequence sum of log((1 - beta_t <d_t, k_t^2>)^2) equals the
    sum of log(f_t(S_t) / f_t(S_before)) measured on the Phase 2 states
    (theorem 5.2's token-local ratios; S_before = alpha_t S_{t-1} when gated)."""
    x = rand_case(T=30, K=6, V=5, apf=True, gated=gated, s0=True, seed=12)
    eta = 0.3
    total = 0.0
    for t, (d, S_prev, S_new, kt, o) in enumerate(step_states(x, eta)):
        k, v = x["k"][0, 0, t], x["v"][0, 0, t]
        al = x["alpha"][0, 0, t] if gated else 1.0
        total += np.log(f_loss(S_new, k, v) / f_loss(al * S_prev, k, v))
    sl = lambda a: None if a is None else a[:1, :1]
    _, _, lr = oracle.precond_scan(sl(x["k"]), sl(x["beta"]), sl(x["r"]), eta, None,
                                   log_ratio=True)
    assert lr.shape == (1, 1)
    assert abs(lr[0, 0] - total) <= 1e-9 * max(1.0, abs(total))


def test_pin_log_ratio_plain_deltanet_closed_form():
    """With d = 1 fixed (eta = 0, r = 1) the ratio of token t is
    (1 - beta_t ||k_t||^2)^2, the plain delta rule's contraction factor."""
    x = rand_case(B=2, H=3, T=50, K=8, V=4, seed=13)
    _, _, lr = oracle.precond_scan(x["k"], x["beta"], None, 0.0, None, log_ratio=True)
    n = np.sum(x["k"] ** 2, axis=-1)
    want = np.sum(np.log((1.0 - x["beta"] * n) ** 2), axis=-1)
    assert np.allclose(lr, want, rtol=1e-12, atol=1e-12)
    # an empty sequence has an empty product
    _, _, lr0 = oracle.precond_scan(x["k"][:, :, :0], x["beta"][:, :, :0], None, 0.1, None,
                                    log_ratio=True)
    assert np.array_equal(lr0, np.zeros((2, 3)))


# ---------------------------------------------------------------------------
# (d) dense unrolled product for T <= 16
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("gated,s0", [(False, False), (True, True)])
def test_pin_d_dense_unrolled_product(gated, s0):
    T, K, V = 16, 6, 4
    x = rand_case(T=T, K=K, V=V, apf=True, gated=gated, s0=s0, seed=3)
    kt, _ = oracle.precond_scan(x["k"], x["beta"], x["r"], 0.2, None)
    o, ST = oracle.delta_fwd(x["q"], x["k"], kt, x["v"], x["beta"], x["alpha"], x["S0"])
    for h in range(2):
        A = []
        for t in range(T):
            al = x["alpha"][0, h, t] if gated else 1.0
            A.append(al * (np.eye(K) - x["beta"][0, h, t] * np.outer(x["k"][0, h, t], kt[0, h, t])))
        S0 = x["S0"][0, h] if s0 else np.zeros((V, K))
        for t in range(T + 1):
            # S_t = S_0 prod_{j<=t} A_j + sum_{i<=t} beta_i v_i ktilde_i^T prod_{i<j<=t} A_j
            P = np.eye(K)
            for j in range(t):
                P = P @ A[j]
            S = S0 @ P
            for i in range(t):
                Q = np.eye(K)
                for j in range(i + 1, t):
                    Q = Q @ A[j]
                S = S + x["beta"][0, h, i] * np.outer(x["v"][0, h, i], kt[0, h, i]) @ Q
            if t >= 1:
                assert np.allclose(o[0, h, t - 1], S @ x["q"][0, h, t - 1], rtol=0, atol=1e-12)
        assert np.allclose(ST[0, h], S, rtol=0, atol=1e-12)


def test_pin_d_dense_affine_preconditioner():
    """Phase 1 as a product of affine maps d -> M_t d + b_t on T <= 16 tokens."""
    T, K = 16, 5
    x = rand_case(T=T, K=K, V=3, apf=True, seed=4)
    eta = 0.25
    d0 = 0.5 + np.arange(2 * K, dtype=np.float64).reshape(1, 2, K) / 7.0
    kt, dT = oracle.precond_scan(x["k"], x["beta"], x["r"], eta, d0)
    for h in range(2):
        M = np.eye(K)
        b = np.zeros(K)
        for t in range(T):
            k, be, r = x["k"][0, h, t], x["beta"][0, h, t], x["r"][0, h, t]
            w = k * k
            n = w.sum()
            dt = M @ d0[0, h] + b
            assert np.allclose(kt[0, h, t], dt * k, rtol=0, atol=1e-13)
            # h_t(d) = ((1 - beta w.d)^2 - 1)/(2n) is quadratic in d; one
            # descent step on it with retention r is affine in d:
            Mt = r * np.eye(K) - eta * be * be * np.outer(w, w) / n
            bt = eta * be * w / n
            M, b = Mt @ M, Mt @ b + bt
        assert np.allclose(dT[0, h], M @ d0[0, h] + b, rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# P5: the step direction is minus the gradient of the DEFINITIONAL surrogate
# ---------------------------------------------------------------------------
def test_pin_p5_descent_direction_by_finite_differences():
    rng = np.random.default_rng(5)
    K, V = 7, 4
    k = rng.standard_normal(K)
    k /= np.linalg.norm(k)
    v = rng.standard_normal(V)
    S = rng.standard_normal((V, K)) * 0.3
    be, eta = 0.7, 0.05
    d = 0.5 + rng.random(K)

    def h_def(dd):
        S_new = S + be * np.outer(v - S @ k, dd * k)
        return (f_loss(S_new, k, v) - f_loss(S, k, v)) / (np.sum((S @ k - v) ** 2) * (k @ k))

    eps = 1e-6
    fd = np.array([(h_def(d + eps * e) - h_def(d - eps * e)) / (2 * eps) for e in np.eye(K)])
    kt, dT = oracle.precond_scan(k[None, None, None], np.array([[[be]]]), None, eta, d[None, None])
    step = (dT[0, 0] - d) / eta                  # r = 1: d_{t+1} - d_t = -eta grad
    assert np.allclose(step, -fd, rtol=1e-6, atol=1e-8)
    # and a small descent step lowers the surrogate it descends
    assert h_def(dT[0, 0]) < h_def(d)


# ---------------------------------------------------------------------------
# P6: gated Newton condition beta <d, k^2> = 1 interpolates exactly
# ---------------------------------------------------------------------------
def test_pin_p6_newton_condition_interpolates():
    rng = np.random.default_rng(6)
    K, V = 8, 6
    k = rng.standard_normal(K)
    k /= np.linalg.norm(k)
    v = rng.standard_normal(V)
    S0 = rng.standard_normal((V, K))
    be = 0.6
    # d0 = c * 1 with beta c ||k||^2 = 1
    d0 = np.full(K, 1.0 / (be * (k @ k)))
    kt, _ = oracle.precond_scan(k[None, None, None], np.array([[[be]]]), None, 0.1, d0[None, None])
    _, ST = oracle.delta_fwd(k[None, None, None], k[None, None, None], kt, v[None, None, None],
                             np.array([[[be]]]), None, S0[None, None])
    assert np.allclose(ST[0, 0] @ k, v, rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# P7: one-hot keys have a closed form (stored fixture, exact rationals)
# ---------------------------------------------------------------------------
def _read_fixture(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, rhs = line.split("=", 1)
                vals[key.strip()] = rhs.split()
    return vals


def test_pin_p7_one_hot_closed_form_fixture():
    fx = _read_fixture("one_hot_apf_closed_form.txt")
    K = int(fx["K"][0])
    beta = float(fractions.Fraction(fx["beta"][0]))
    eta = float(fractions.Fraction(fx["eta"][0]))
    hits = [int(i) for i in fx["hits"]]
    r = [float(fractions.Fraction(s)) for s in fx["r"]]
    d0 = np.array([float(fractions.Fraction(s)) for s in fx["d0"]])
    want = np.array([float(fractions.Fraction(s)) for s in fx["dT"]])
    T = len(hits)
    k = np.zeros((1, 1, T, K))
    k[0, 0, np.arange(T), hits] = 1.0
    kt, dT = oracle.precond_scan(k, np.full((1, 1, T), beta), np.array(r)[None, None], eta,
                                 d0[None, None])
    assert np.allclose(dT[0, 0], want, rtol=1e-14, atol=0)


def test_pin_p7_one_hot_geometric_approach_to_inverse_beta():
    # r = 1: after m hits on coordinate i, d_i = 1/beta - (1/beta - d0_i)(1 - eta beta^2)^m
    K, beta, eta, m = 4, 0.8, 0.3, 50
    k = np.zeros((1, 1, m, K))
    k[0, 0, :, 2] = 1.0
    d0 = np.array([0.3, 1.7, 0.2, 2.5])
    _, dT = oracle.precond_scan(k, np.full((1, 1, m), beta), None, eta, d0[None, None])
    want = d0.copy()
    want[2] = 1 / beta - (1 / beta - d0[2]) * (1 - eta * beta ** 2) ** m
    assert np.allclose(dT[0, 0], want, rtol=1e-13, atol=0)


# ---------------------------------------------------------------------------
# P8: eta = 0 leaves only the retention: d_t = (prod_{j<t} r_j) d_0
# ---------------------------------------------------------------------------
def test_pin_p8_eta_zero_is_pure_retention():
    x = rand_case(T=30, K=5, V=3, apf=True, seed=8)
    kt, dT = oracle.precond_scan(x["k"], x["beta"], x["r"], 0.0, None)
    rho = np.concatenate([np.ones((1, 2, 1)), np.cumprod(x["r"], axis=-1)], axis=-1)
    assert np.allclose(kt, rho[..., :-1, None] * x["k"], rtol=1e-14, atol=0)
    assert np.allclose(dT, np.broadcast_to(rho[..., -1:], dT.shape), rtol=1e-14, atol=0)


# ---------------------------------------------------------------------------
# P9: state chaining -- [0,T) equals [0,T1) then [T1,T) with (d, S) carried
# ---------------------------------------------------------------------------
def test_pin_p9_state_chaining():
    x = rand_case(B=1, H=3, T=50, K=6, V=5, apf=True, gated=True, s0=True, seed=9)
    kt, dT, o, ST = oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["r"], 0.2, None,
                                   x["alpha"], x["S0"])
    T1 = 17
    a = lambda t, lo, hi: t[:, :, lo:hi]
    kt1, dT1, o1, ST1 = oracle.forward(a(x["q"], 0, T1), a(x["k"], 0, T1), a(x["v"], 0, T1),
                                       a(x["beta"], 0, T1), a(x["r"], 0, T1), 0.2, None,
                                       a(x["alpha"], 0, T1), x["S0"])
    kt2, dT2, o2, ST2 = oracle.forward(a(x["q"], T1, 50), a(x["k"], T1, 50), a(x["v"], T1, 50),
                                       a(x["beta"], T1, 50), a(x["r"], T1, 50), 0.2, dT1,
                                       a(x["alpha"], T1, 50), ST1)
    assert np.array_equal(np.concatenate([kt1, kt2], 2), kt)
    assert np.array_equal(np.concatenate([o1, o2], 2), o)
    assert np.array_equal(dT2, dT) and np.array_equal(ST2, ST)


# ---------------------------------------------------------------------------
# degenerate inputs
# ---------------------------------------------------------------------------
def test_zero_key_leaves_d_to_retention_and_state_to_decay():
    K, V = 4, 3
    k = np.zeros((1, 1, 1, K))
    d0 = np.array([[[1.0, 2.0, 3.0, 4.0]]])
    kt, dT = oracle.precond_scan(k, np.array([[[0.5]]]), np.array([[[0.9]]]), 0.2, d0)
    assert np.array_equal(kt, np.zeros_like(kt))
    assert np.allclose(dT, 0.9 * d0, rtol=1e-15, atol=0)
    S0 = np.arange(V * K, dtype=np.float64).reshape(1, 1, V, K)
    q = np.ones((1, 1, 1, K))
    o, ST = oracle.delta_fwd(q, k, kt, np.ones((1, 1, 1, V)), np.array([[[0.5]]]),
                             np.array([[[0.75]]]), S0)
    assert np.allclose(ST, 0.75 * S0, rtol=1e-15, atol=0)
    assert np.allclose(o[0, 0, 0], (0.75 * S0[0, 0]) @ q[0, 0, 0], rtol=1e-15, atol=0)


def test_empty_sequence_returns_initial_state():
    d0 = np.array([[[1.5, 0.5]]])
    kt, dT = oracle.precond_scan(np.zeros((1, 1, 0, 2)), np.zeros((1, 1, 0)), None, 0.1, d0)
    assert kt.shape == (1, 1, 0, 2) and np.array_equal(dT, d0)
    S0 = np.ones((1, 1, 3, 2))
    o, ST = oracle.delta_fwd(np.zeros((1, 1, 0, 2)), np.zeros((1, 1, 0, 2)),
                             np.zeros((1, 1, 0, 2)), np.zeros((1, 1, 0, 3)),
                             np.zeros((1, 1, 0)), None, S0)
    assert o.shape == (1, 1, 0, 3) and np.array_equal(ST, S0)


def test_descent_keeps_contraction_where_ascent_diverges():
    """The reading of the APF sign: with the descent step |1 - beta a_t| stays
    below 1 on a long normalised stream; the printed '+' sign would not."""
    x = rand_case(B=1, H=1, T=4000, K=32, V=2, seed=10)
    k, be = x["k"], x["beta"]
    kt, _ = oracle.precond_scan(k, be, None, 0.1, None)
    d = kt / k
    a = np.sum(d * k * k, axis=-1)
    assert np.max(np.abs(1 - be * a)) < 1.0
    # ascent = descent with eta -> -eta
    kt2, _ = oracle.precond_scan(k, be, None, -0.1, None)
    a2 = np.sum((kt2 / k) * k * k, axis=-1)
    assert np.max(np.abs(1 - be * a2)) > 1.0
