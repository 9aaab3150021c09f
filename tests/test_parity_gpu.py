"""GPU-vs-oracle parity through the C ABI.

Every output of both phases (ktilde, d_T, o, S_T) is compared element by
element with the fp64 oracle on the same seeded inputs, within the
normwise tolerance of the I/O type (1e-4 fp32, 2e-2 bf16).  The five named
workloads run at full size on the GPU; the oracle checks a sample of their
sequences.  Small shapes cover every chunk-tail case and the optional
inputs.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
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


def run_gpu(x, ws=None):
    g = to_cuda(x)
    ws = ws or ops.Workspace()
    kt, dT, o, ST = ops.forward(g["q"], g["k"], g["v"], g["beta"], g["r"], g["eta"], g["d0"],
                                g["alpha"], g["S0"], workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0, ops.status_string(ws.status())
    return kt, dT, o, ST


def check_all(x, io, heads=None, label=""):
    kt, dT, o, ST = run_gpu(x)
    okt, odT, oo, oST = oracle_forward(x, heads)
    sel = (lambda t: pick(t, heads)) if heads is not None else (lambda t: t)
    tol = TOL[io]
    errs = {"ktilde": rel_err(sel(kt), okt), "dT": rel_err(sel(dT), odT),
            "o": rel_err(sel(o), oo), "ST": rel_err(sel(ST), oST)}
    for name, e in errs.items():
        assert e <= tol, "%s %s: %.3e > %.1e (%s)" % (label, name, e, tol, errs)
    # Phase 2 alone, fed the GPU's own (io-rounded) ktilde
    xs = synth.slice_heads(x, heads) if heads is not None else x
    o2, ST2 = oracle.delta_fwd(xs["q"], xs["k"], sel(kt).cpu(), xs["v"], xs["beta"],
                               xs["alpha"], xs["S0"])
    assert rel_err(sel(o), o2) <= tol and rel_err(sel(ST), ST2) <= tol, label
    return errs


@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_workload_parity_full_size(name):
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w)
    BH = w.B * w.H
    heads = None if BH * w.T <= 4096 else sorted({0, BH // 2, BH - 1})
    errs = check_all(x, w.io, heads, name)
    print(name, {k: "%.2e" % v for k, v in errs.items()})


SHAPES = [1, 15, 63, 64, 65, 127, 200]


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("T", SHAPES)
def test_chunk_tails(io, T):
    for K, V in itertools.product([64, 128], [64, 128]):
        x = synth.make_random(2, 3, T, K, V, io=io, apf=True, gated=(T % 2 == 1), s0=True,
                              d0=True, seed=T + K + V)
        check_all(x, io, None, "%s T=%d K=%d V=%d" % (io, T, K, V))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_optional_inputs_null(io):
    # r, alpha, S0, d0 all NULL: the plain OSDN recurrence from d0 = 1, S0 = 0
    x = synth.make_random(1, 4, 300, 128, 64, io=io, seed=11)
    check_all(x, io, None, "null optionals")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_state_chaining_on_gpu(io):
    x = synth.make_random(1, 2, 400, 64, 128, io=io, apf=True, gated=True, s0=True, seed=12)
    g = to_cuda(x)
    kt, dT, o, ST = ops.forward(g["q"], g["k"], g["v"], g["beta"], g["r"], g["eta"], None,
                                g["alpha"], g["S0"])
    T1 = 137
    cut = lambda t, lo, hi: t[:, :, lo:hi].contiguous()
    kt1, dT1, o1, ST1 = ops.forward(cut(g["q"], 0, T1), cut(g["k"], 0, T1), cut(g["v"], 0, T1),
                                    cut(g["beta"], 0, T1), cut(g["r"], 0, T1), g["eta"], None,
                                    cut(g["alpha"], 0, T1), g["S0"])
    kt2, dT2, o2, ST2 = ops.forward(cut(g["q"], T1, 400), cut(g["k"], T1, 400),
                                    cut(g["v"], T1, 400), cut(g["beta"], T1, 400),
                                    cut(g["r"], T1, 400), g["eta"], dT1,
                                    cut(g["alpha"], T1, 400), ST1)
    tol = TOL[io]
    assert rel_err(torch.cat([kt1, kt2], 2), kt.double().cpu().numpy()) <= tol
    assert rel_err(torch.cat([o1, o2], 2), o.double().cpu().numpy()) <= tol
    assert rel_err(dT2, dT.double().cpu().numpy()) <= tol
    assert rel_err(ST2, ST.double().cpu().numpy()) <= tol


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_deterministic_bitwise(io):
    x = synth.make_random(2, 2, 333, 128, 128, io=io, apf=True, gated=True, s0=True, seed=13)
    a = run_gpu(x)
    b = run_gpu(x)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_empty_sequence_copies_initial_state(io):
    x = synth.make_random(1, 3, 0, 64, 64, io=io, s0=True, d0=True, seed=14)
    g = to_cuda(x)
    kt, dT, o, ST = ops.forward(g["q"], g["k"], g["v"], g["beta"], None, 0.1, g["d0"], None,
                                g["S0"])
    torch.cuda.synchronize()
    assert torch.equal(dT, g["d0"]) and torch.equal(ST, g["S0"])
    assert kt.numel() == 0 and o.numel() == 0


def test_alias_rejected_before_launch():
    x = to_cuda(synth.make_random(1, 1, 16, 64, 64, io="bf16", seed=15))
    with pytest.raises(ops.OsdnError) as ei:
        ops.precond_scan(x["k"], x["beta"], ktilde=x["k"])
    assert ei.value.code == -9


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("case", ["converging", "slow_retention", "expansive_token", "expansive_step",
                                  "short_tail"])
def test_segmented_scan_exact(io, case):
    """The time-segmented scan (used when a retention gate is given) equals the
    token recurrence whether the speculative segment starts verify or must be
    recomputed."""
    T = 3001 if case == "short_tail" else 3000
    x = synth.make_random(1, 4, T, 128, 64, io=io, apf=True, d0=True, seed=21)
    if case == "slow_retention":      # warm-up cannot forget the guess: every start is repaired
        x["r"] = torch.full_like(x["r"], 0.99995)
    if case == "expansive_token":     # one map with ||A_t|| > 1: all segments recomputed
        x["r"][:, :, 1700] = 1.5
    if case == "expansive_step":      # |r_t - eta beta_t^2 |w_t|^2 / n_t| > 1 at one token
        x["eta"] = 2.5
        x["k"][:, :, 1700] = 0.0
        x["k"][:, :, 1700, 5] = 1.0
        x["beta"][:, :, 1700] = 1.0
    g = to_cuda(x)
    ws = ops.Workspace()
    kt, dT = ops.precond_scan(g["k"], g["beta"], g["r"], g["eta"], g["d0"], workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    okt, odT = oracle.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"])
    tol = TOL[io]
    assert rel_err(kt, okt) <= tol, rel_err(kt, okt)
    assert rel_err(dT, odT) <= tol, rel_err(dT, odT)


def test_segmented_scan_many_accepted_segments_fp32():
    """Many speculative segments whose starts are accepted, with the slowest
    retention that still passes the check: r in [0.87, 0.90], so that the
    128-token warm-up leaves a start about 2^-22.6 off, just inside the 2^-21
    acceptance bound.  The differences of the 32 accepted segments carry
    through the scan, and the result must still hold the fp32 tolerance on
    ktilde and d_T."""
    T = 8192
    x = synth.make_random(1, 2, T, 128, 64, io="f32", apf=True, d0=True, seed=22)
    g = torch.Generator().manual_seed(23)
    x["r"] = (0.87 + 0.03 * torch.rand(x["r"].shape, generator=g)).contiguous()
    nseg = T // 256
    assert ops.precond_scan_workspace_bytes(1, 2, T, 128) >= 256 + 2 * nseg * 128 * 8
    gx = to_cuda(x)
    ws = ops.Workspace()
    kt, dT = ops.precond_scan(gx["k"], gx["beta"], gx["r"], gx["eta"], gx["d0"], workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    okt, odT = oracle.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"])
    assert rel_err(kt, okt) <= 1e-4, rel_err(kt, okt)
    assert rel_err(dT, odT) <= 1e-4, rel_err(dT, odT)


@pytest.mark.parametrize("nfull", [128, 256 + 64])
def test_phase2_slabs_with_ragged_last_slab(nfull):
    # nfull chunks of 64 tokens and a ragged one: without a decay the bf16
    # Phase 2 runs them as slabs of 64 chunks and a last one of 1 chunk,
    # preparing later slabs while earlier ones run and carrying the state
    # between slabs; S0 and S_T cross the slab seams
    T = 64 * nfull + 37
    x = synth.make_random(1, 2, T, 64, 64, io="bf16", apf=True, gated=False, s0=True, d0=True,
                          seed=21)
    check_all(x, "bf16", None, "slabs T=%d" % T)


@pytest.mark.parametrize("case", ["accepted", "all_repaired", "one_repaired", "ragged",
                                  "wide_rows"])
def test_phase2_time_segments_with_decay(case):
    # With a decay the bf16 chain runs in time segments (here 3 of 16 chunks):
    # every segment but the first starts from a zero state 4 chunks early, and
    # a start that does not match its predecessor's end is recomputed.
    # accepted: the synthetic decay forgets the warm-up's guess; all_repaired:
    # a decay of 0.9999 does not, every later segment is recomputed;
    # one_repaired: no decay over the first segment's last 4 chunks, so only
    # the second segment's start is off; ragged: a ragged last chunk and
    # segment; wide_rows: K = V = 128 (two CTAs of 64 value rows a sequence,
    # each deciding for its own rows)
    K = V = 128 if case == "wide_rows" else 64
    T = 64 * 51 + 17 if case == "ragged" else 64 * 48
    x = synth.make_random(1, 2, T, K, V, io="bf16", apf=True, gated=True, s0=True, d0=True,
                          seed=41)
    if case == "all_repaired":
        x["alpha"] = torch.full_like(x["alpha"], 0.9999)
    if case == "one_repaired":
        x["alpha"][:, :, 64 * 12:64 * 16] = 1.0
    check_all(x, "bf16", None, "segments %s" % case)


def test_concurrent_calls_share_the_library_streams():
    # two host threads, two streams, multi-slab calls at once: the results
    # equal those of the same calls made one after the other
    import threading
    xs = [synth.make_random(1, 2, 4096 + 100 * i, 128, 128, io="bf16", apf=True, gated=(i == 1),
                            s0=True, seed=30 + i) for i in range(2)]
    gs = [to_cuda(x) for x in xs]
    ref = [run_gpu(x) for x in xs]
    out = [None, None]

    def work(i):
        s = torch.cuda.Stream()
        g = gs[i]
        with torch.cuda.stream(s):
            ws = ops.Workspace(stream=s)
            out[i] = ops.forward(g["q"], g["k"], g["v"], g["beta"], g["r"], g["eta"], g["d0"],
                                 g["alpha"], g["S0"], workspace=ws, stream=s)
        s.synchronize()
        assert ws.status(s) == 0

    th = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    for i in range(2):
        for a, b in zip(out[i], ref[i]):
            assert torch.equal(a, b), "thread %d" % i


@pytest.mark.parametrize("bad", ["alpha_zero", "alpha_negative", "beta_nan"])
def test_invalid_gates_reported_by_the_device(bad):
    # the bf16 chunk pass takes log alpha: a decay that is not positive (or a
    # beta that is not finite) is recorded in the status word as
    # OSDN_ERR_DEVICE; nothing faults and the next call is clean
    x = synth.make_random(1, 2, 200, 64, 64, io="bf16", apf=True, gated=True, seed=51)
    g = to_cuda(x)
    if bad == "alpha_zero":
        g["alpha"][0, 1, 70] = 0.0
    if bad == "alpha_negative":
        g["alpha"][0, 0, 3] = -0.5
    if bad == "beta_nan":
        g["beta"][0, 1, 199] = float("nan")
    ws = ops.Workspace()
    kt, _ = ops.precond_scan(g["k"], g["beta"].nan_to_num(0.5), g["r"], g["eta"])
    ops.chunk_fwd(g["q"], g["k"], kt, g["v"], g["beta"], g["alpha"], g["S0"], workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == -8, ops.status_string(ws.status())
    ws2 = ops.Workspace()
    run_gpu(x, ws2)


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_more_sequences_than_one_grid_dimension_holds(io):
    # 65,537 sequences: the kernels spread sequences over two grid dimensions,
    # so the first, the 65,535th and the last one are all computed
    x = synth.make_random(1, 65537, 70, 64, 64, io=io, apf=True, gated=(io == "bf16"), s0=True,
                          seed=61)
    kt, dT, o, ST = run_gpu(x)
    heads = [0, 65534, 65535, 65536]
    okt, odT, oo, oST = oracle_forward(x, heads)
    tol = TOL[io]
    for name, got, want in (("ktilde", kt, okt), ("dT", dT, odT), ("o", o, oo), ("ST", ST, oST)):
        assert rel_err(pick(got, heads), want) <= tol, name
