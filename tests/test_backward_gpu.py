"""osdn_backward (the gradients of both phases) against the fp64 reference
gradients of ``oracle.backward`` (autograd through a token-by-token
restatement of the forward, pinned by finite differences of the C oracle).

Every input's gradient is compared with the normwise tolerance of the I/O
type: q, k, v, beta, r, alpha, d0, S0 and eta (the sum of the per-sequence
shares).  The kernels take ktilde as the forward stored it; here it is the
oracle's Phase 1 output rounded to the I/O type, and the reference is the
exact derivative given that same stored ktilde (the straight-through option
of ``oracle.backward``), so that the comparison is about the backward alone.
(Against the derivative with the exact ktilde, the bf16 rounding of ktilde
alone moves the eta gradient of an 8192-token head by about 1.6e-2: its sum
over tokens cancels heavily.)  Cases cover both I/O types, every (K, V) pair,
one and several 16-token sub-chunks with ragged tails, T = 1 and T = 0,
optional inputs and cotangents left out, a zero key, the time segments of
the Phase 1 adjoint (accepted, repaired, all recomputed), and determinism;
and the full shape the benchmark times, with its last head checked.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward
from preconditioned_delta_rule_phase1_gb300 import build as osdn_build
from preconditioned_delta_rule_phase1_gb300 import ops, synth
from tests._util import TOL, rel_err, to_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    osdn_build.build()
    ops.lib()


def cotangents(B, H, T, K, V, io, seed, which=("o", "ST", "dT", "kt")):
    g = torch.Generator().manual_seed(seed)
    dt = synth.torch_dtype(io)
    c = {"o": torch.randn(B, H, T, V, generator=g).to(dt),
         "ST": torch.randn(B, H, V, K, generator=g),
         "dT": torch.randn(B, H, K, generator=g),
         "kt": torch.randn(B, H, T, K, generator=g).to(dt)}
    return {n: (c[n].contiguous() if n in which else None) for n in c}


def ktilde_of(x):
    kt, _ = oracle.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"])
    return torch.from_numpy(np.asarray(kt)).to(x["k"].dtype).contiguous()


def run(x, cot, kt=None):
    kt = ktilde_of(x) if kt is None else kt
    g = to_cuda(x)
    c = to_cuda(cot)
    got = ops.backward(g["q"], g["k"], kt.cuda(), g["v"], g["beta"], g["r"], g["eta"], g["d0"],
                       g["alpha"], g["S0"], do=c["o"], dST=c["ST"], ddT=c["dT"],
                       dktilde=c["kt"])
    torch.cuda.synchronize()
    return got


def reference(x, cot, kt):
    # the exact derivative given the stored ktilde the kernels receive
    return backward.grads(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"],
                          x["alpha"], x["S0"], do=cot["o"], ddT=cot["dT"], dST=cot["ST"],
                          dkt=cot["kt"], ktilde=kt)


def check(x, cot, io):
    kt = ktilde_of(x)
    got = run(x, cot, kt)
    ref = reference(x, cot, kt)
    assert set(got) == set(ref), (sorted(got), sorted(ref))
    errs = {}
    for n, r in ref.items():
        val = got[n].double().sum().item() if n == "eta" else got[n]
        errs[n] = rel_err(torch.tensor(val) if n == "eta" else val, np.asarray(r))
    assert max(errs.values()) <= TOL[io], errs
    return errs


CASES = [
    # io, K, V, T, gated, apf
    ("f32", 64, 64, 100, True, True),      # six sub-chunks and a tail of 4
    ("f32", 128, 128, 37, False, True),
    ("f32", 128, 64, 5, True, True),       # shorter than one sub-chunk
    ("f32", 64, 128, 16, True, False),     # exactly one sub-chunk, no retention gate
    ("bf16", 128, 128, 100, True, True),
    ("bf16", 64, 128, 33, True, True),
    ("bf16", 128, 64, 1, False, True),
    ("bf16", 64, 64, 48, True, True),
]


@pytest.mark.parametrize("io,K,V,T,gated,apf", CASES)
def test_gradients_match_reference(io, K, V, T, gated, apf):
    x = synth.make_random(1, 2, T, K, V, io=io, apf=apf, gated=gated, s0=True, d0=True,
                          seed=400 + T + K)
    check(x, cotangents(1, 2, T, K, V, io, 500 + T), io)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_optional_inputs_and_cotangents_left_out(io):
    # r, d0, alpha, S0 at their defaults; only the output's cotangent given
    x = synth.make_random(2, 1, 50, 64, 64, io=io, seed=61)
    assert x["r"] is None and x["alpha"] is None and x["S0"] is None and x["d0"] is None
    errs = check(x, cotangents(2, 1, 50, 64, 64, io, 62, which=("o",)), io)
    assert set(errs) == {"q", "k", "v", "beta", "eta"}


def test_a_zero_key():
    x = synth.make_random(1, 2, 40, 64, 64, io="f32", apf=True, gated=True, s0=True, d0=True,
                          seed=71)
    x["k"][0, 1, 7] = 0.0
    x["k"][0, 0, 39] = 0.0
    check(x, cotangents(1, 2, 40, 64, 64, "f32", 72), "f32")


def test_longer_sequence():
    x = synth.make_random(1, 2, 700, 128, 128, io="bf16", apf=True, gated=True, s0=True,
                          seed=81)
    check(x, cotangents(1, 2, 700, 128, 128, "bf16", 82), "bf16")


@pytest.mark.parametrize("io,T", [("f32", 1025), ("bf16", 2048), ("f32", 2100)])
def test_reverse_sweep_windows(io, T):
    # the state adjoint's reverse sweep runs in windows of 1024 tokens, the
    # state gradient carried between them: a last window of one token, two
    # full windows, and a ragged third one
    x = synth.make_random(1, 2, T, 64, 64, io=io, apf=True, gated=True, s0=True, d0=True,
                          seed=90 + T)
    check(x, cotangents(1, 2, T, 64, 64, io, 91 + T), io)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("case", ["accepted", "slow_retention", "expansive_token"])
def test_phase1_adjoint_time_segments(io, case):
    # with a retention gate the Phase 1 adjoint runs in time segments of 256
    # tokens, each started from lam = 0 128 tokens past its end and verified
    # against its successor's exact start: accepted as is, every start
    # repaired (a retention of 0.99995 forgets nothing in 128 tokens), or
    # every segment recomputed (one step map with norm above 1)
    x = synth.make_random(1, 2, 1500, 64, 64, io=io, apf=True, gated=True, s0=True, d0=True,
                          seed=101)
    if case == "slow_retention":
        x["r"] = torch.full_like(x["r"], 0.99995)
    if case == "expansive_token":
        x["r"][:, :, 900] = 1.5
    check(x, cotangents(1, 2, 1500, 64, 64, io, 102), io)


def test_deterministic():
    x = synth.make_random(2, 2, 90, 128, 64, io="bf16", apf=True, gated=True, s0=True, d0=True,
                          seed=91)
    cot = cotangents(2, 2, 90, 128, 64, "bf16", 92)
    kt = ktilde_of(x)
    a, b = run(x, cot, kt), run(x, cot, kt)
    for n in a:
        assert torch.equal(a[n], b[n]), n


def test_empty_sequence():
    x = synth.make_random(1, 2, 0, 64, 64, io="f32", apf=True, gated=True, s0=True, d0=True,
                          seed=93)
    cot = cotangents(1, 2, 0, 64, 64, "f32", 94)
    got = run(x, cot, kt=torch.empty(1, 2, 0, 64))
    assert torch.equal(got["S0"].cpu(), cot["ST"])
    assert torch.equal(got["d0"].cpu(), cot["dT"])
    assert torch.equal(got["eta"].cpu(), torch.zeros(1, 2))
    for n in ("q", "k", "v", "beta", "r", "alpha"):
        assert got[n].numel() == 0


def test_full_size_sampled_head():
    # the shape `bench.py --backward` times (2 x 16 heads x 8192 tokens,
    # d_k = d_v = 128, bf16, adaptive forgetting), output cotangent given;
    # the last head (the largest offsets) against the reference gradients --
    # heads are independent, so the sample is exact
    w = synth.WORKLOADS["lm1p3b_apf_bf16"]
    x = synth.make_inputs(w)
    gen = torch.Generator().manual_seed(1)
    dO = torch.randn(w.B, w.H, w.T, w.V, generator=gen).to(x["v"].dtype)
    kt = ktilde_of(x)
    got = run(x, {"o": dO, "ST": None, "dT": None, "kt": None}, kt)
    head = w.B * w.H - 1
    xs = synth.slice_heads(x, [head])
    ref = backward.grads(xs["q"], xs["k"], xs["v"], xs["beta"], xs["r"], xs["eta"], xs["d0"],
                         xs["alpha"], xs["S0"], do=dO.reshape(-1, w.T, w.V)[head][None, None],
                         ktilde=kt.reshape(-1, w.T, w.K)[head][None, None])
    assert set(got) == set(ref), (sorted(got), sorted(ref))
    errs = {}
    for n, r in ref.items():
        flat = got[n].reshape(-1, *got[n].shape[2:])[head]   # eta: this head's share
        errs[n] = rel_err(flat, np.reshape(r, flat.shape))
    assert max(errs.values()) <= TOL["bf16"], errs
