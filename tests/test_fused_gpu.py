"""osdn_forward: both phases in one call, with ktilde kept off global memory
for bf16 I/O.

The preconditioner scan then writes, instead of ktilde, the coefficient e_t
of every token and d at every 64-token boundary, and the chunk preparation
rebuilds each chunk's ktilde on chip as (rho d_c + P W) . K.  Every output
(o, d_T, S_T) is compared with the fp64 oracle within the I/O tolerance and
d_T bit for bit with the two-call path (the scan's arithmetic is the same).
The rebuilt preconditioner differs from the scan's own by about 2^-16
relative, so the fused path must be as accurate as the two-call path: its
error against the oracle may exceed the two-call path's by at most a
quarter of the tolerance (the bf16 roundings downstream of ktilde differ
between the two, so they are not compared with each other directly).  The
scan's checkpoints themselves (e_t and d every 64 tokens, in the workspace)
are compared with the oracle's scan at the fp32 tolerance.
"""
import itertools

import numpy as np
import pytest
import torch

from preconditioned_delta_rule_phase1_gb300 import build as osdn_build
from preconditioned_delta_rule_phase1_gb300 import ops, synth
from tests._util import TOL, oracle_forward, pick, rel_err, to_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    osdn_build.build()
    ops.lib()


def run_fused(g, ws=None):
    ws = ws or ops.Workspace()
    dT, o, ST = ops.forward_fused(g["q"], g["k"], g["v"], g["beta"], g["r"], g["eta"], g["d0"],
                                  g["alpha"], g["S0"], workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0, ops.status_string(ws.status())
    return dT, o, ST


def run_two_calls(g):
    ws = ops.Workspace()
    _, dT, o, ST = ops.forward(g["q"], g["k"], g["v"], g["beta"], g["r"], g["eta"], g["d0"],
                               g["alpha"], g["S0"], workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0, ops.status_string(ws.status())
    return dT, o, ST


def check_fused(x, io, heads=None, label=""):
    g = to_cuda(x)
    dT, o, ST = run_fused(g)
    _, odT, oo, oST = oracle_forward(x, heads)
    sel = (lambda t: pick(t, heads)) if heads is not None else (lambda t: t)
    tol = TOL[io]
    errs = {"dT": rel_err(sel(dT), odT), "o": rel_err(sel(o), oo), "ST": rel_err(sel(ST), oST)}
    for name, e in errs.items():
        assert e <= tol, "%s %s: %.3e > %.1e (%s)" % (label, name, e, tol, errs)
    dT2, o2, ST2 = run_two_calls(g)
    assert torch.equal(dT, dT2), label
    if io == "f32":   # the same two kernels, ktilde kept in the workspace
        assert torch.equal(o, o2) and torch.equal(ST, ST2), label
    else:
        e2 = {"o": rel_err(sel(o2), oo), "ST": rel_err(sel(ST2), oST)}
        for name in ("o", "ST"):
            assert errs[name] <= e2[name] + tol / 4, "%s %s: fused %.3e, two calls %.3e" % (
                label, name, errs[name], e2[name])
        errs.update(two_call_o=e2["o"], two_call_ST=e2["ST"])
    return errs


@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_fused_workload_parity_full_size(name):
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w)
    BH = w.B * w.H
    heads = None if BH * w.T <= 4096 else sorted({0, BH // 2, BH - 1})
    errs = check_fused(x, w.io, heads, name)
    print(name, {k: "%.2e" % v for k, v in errs.items()})


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 15, 63, 64, 65, 127, 200])
def test_fused_chunk_tails(io, T):
    for K, V in itertools.product([64, 128], [64, 128]):
        x = synth.make_random(2, 3, T, K, V, io=io, apf=True, gated=(T % 2 == 1), s0=True,
                              d0=True, seed=T + K + V)
        check_fused(x, io, None, "%s T=%d K=%d V=%d" % (io, T, K, V))


@pytest.mark.parametrize("H", [4, 400])
def test_fused_without_retention(H):
    # no retention gate: one scan segment a sequence -- a CTA per sequence for
    # few sequences (H = 4), one warp per sequence for many (H = 400)
    x = synth.make_random(1, H, 300, 128, 64, io="bf16", d0=True, seed=70 + H)
    heads = sorted({0, H // 2, H - 1})
    check_fused(x, "bf16", heads, "no retention H=%d" % H)


@pytest.mark.parametrize("case", ["slow_retention", "expansive_token"])
def test_fused_after_scan_repairs(case):
    # the scan's speculative segments are recomputed (every one, or all after
    # one expanding token): the repairs rewrite e_t and the checkpoints too
    x = synth.make_random(1, 4, 3000, 128, 64, io="bf16", apf=True, d0=True, seed=21)
    if case == "slow_retention":
        x["r"] = torch.full_like(x["r"], 0.99995)
    if case == "expansive_token":
        x["r"][:, :, 1700] = 1.5
    check_fused(x, "bf16", None, case)


@pytest.mark.parametrize("case", ["slabs", "decay_segments", "decay_segments_repaired"])
def test_fused_phase2_schedules(case):
    # the chunk preparation runs in slabs overlapped with the chain, or (with
    # a decay) over every chunk before a time-segmented chain
    if case == "slabs":
        x = synth.make_random(1, 2, 64 * 128 + 37, 64, 64, io="bf16", apf=True, s0=True, d0=True,
                              seed=81)
    else:
        x = synth.make_random(1, 2, 64 * 48, 64, 64, io="bf16", apf=True, gated=True, s0=True,
                              d0=True, seed=82)
        if case == "decay_segments_repaired":
            x["alpha"] = torch.full_like(x["alpha"], 0.9999)
    check_fused(x, "bf16", None, case)


def test_fused_zero_keys():
    # a zero key takes no preconditioner step (e_t = 0) and writes nothing
    x = synth.make_random(1, 3, 250, 128, 128, io="bf16", apf=True, gated=True, s0=True, seed=91)
    x["k"][:, :, 5] = 0.0
    x["k"][:, 1, 64:70] = 0.0
    x["k"][:, 2, 249] = 0.0
    check_fused(x, "bf16", None, "zero keys")


@pytest.mark.parametrize("apf", [True, False])
def test_fused_checkpoints_match_the_oracle_scan(apf):
    # the workspace after the status word: the scan's segment scratch, then
    # e_t [B*H][T] and d every 64 tokens [B*H][ceil(T/64)][K], all fp32
    import oracle
    B, H, T, K, V = 1, 3, 1100, 64, 64
    x = synth.make_random(B, H, T, K, V, io="bf16", apf=apf, d0=True, eta=0.5, seed=95)
    g = to_cuda(x)
    ws = ops.Workspace()
    run_fused(g, ws)
    r256 = lambda n: -(-n // 256) * 256
    off_e = 256 + r256(ops.precond_scan_workspace_bytes(B, H, T, K) - 256)
    off_d = off_e + r256(B * H * T * 4)
    nch = -(-T // 64)
    raw = ws.buf
    e_gpu = raw[off_e:off_e + B * H * T * 4].view(torch.float32).reshape(H, T).double().cpu().numpy()
    d_gpu = raw[off_d:off_d + B * H * nch * K * 4].view(torch.float32).reshape(H, nch, K)
    d_gpu = d_gpu.double().cpu().numpy()
    kt, dT = oracle.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"])
    k = x["k"][0].double().numpy()
    d = np.concatenate([np.asarray(kt)[0] / k, np.asarray(dT)[0][:, None]], axis=1)  # d_0..d_T
    r = np.ones((H, T)) if x["r"] is None else x["r"][0].double().numpy()
    w = k * k
    e = ((d[:, 1:] - r[..., None] * d[:, :-1]) * w).sum(-1) / (w * w).sum(-1)
    assert rel_err(torch.as_tensor(d_gpu), d[:, 0:T:64]) <= TOL["f32"]
    assert rel_err(torch.as_tensor(e_gpu), e) <= TOL["f32"]


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_fused_empty_sequence(io):
    x = synth.make_random(1, 2, 0, 64, 64, io=io, apf=True, s0=True, d0=True, seed=92)
    g = to_cuda(x)
    dT, o, ST = run_fused(g)
    assert o.numel() == 0
    assert torch.equal(dT, g["d0"]) and torch.equal(ST, g["S0"])


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_fused_deterministic_bitwise(io):
    x = synth.make_random(2, 2, 333, 128, 128, io=io, apf=True, gated=True, s0=True, seed=93)
    g = to_cuda(x)
    a = run_fused(g)
    b = run_fused(g)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_fused_more_sequences_than_one_grid_dimension_holds():
    x = synth.make_random(1, 65537, 70, 64, 64, io="bf16", apf=True, gated=True, s0=True,
                          seed=94)
    g = to_cuda(x)
    dT, o, ST = run_fused(g)
    heads = [0, 65534, 65535, 65536]
    _, odT, oo, oST = oracle_forward(x, heads)
    for name, got, want in (("dT", dT, odT), ("o", o, oo), ("ST", ST, oST)):
        assert rel_err(pick(got, heads), want) <= TOL["bf16"], name
