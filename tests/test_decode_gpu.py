"""The recurrent decode step (osdn_decode_step) against the fp64 oracle.

One step must equal both phases of the oracle on a sequence of length 1
from the same (d, S); twenty chained steps must equal the oracle on the
twenty-token sequence.  All of d, S (updated in place), o and ktilde are
compared, within the normwise tolerance of the I/O type.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from preconditioned_delta_rule_phase1_gb300 import build as osdn_build
from preconditioned_delta_rule_phase1_gb300 import ops, synth
from tests._util import TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    osdn_build.build()
    ops.lib()


def oracle_steps(x, d0, S0):
    kt, dT = oracle.precond_scan(x["k"], x["beta"], x["r"], x["eta"], d0)
    o, ST = oracle.delta_fwd(x["q"], x["k"], kt, x["v"], x["beta"], x["alpha"], S0)
    return np.asarray(kt), np.asarray(dT), np.asarray(o), np.asarray(ST)


def run_steps(x, d0, S0):
    dev = lambda t: None if t is None else t.cuda()
    d = d0.clone().cuda()
    S = S0.clone().cuda()
    T = x["k"].shape[2]
    os_, kts = [], []
    ws = ops.Workspace()
    for t in range(T):
        sl = lambda n: None if x[n] is None else x[n][:, :, t].contiguous().cuda()
        o, kt = ops.decode_step(sl("q"), sl("k"), sl("v"), sl("beta"), d, S, r=sl("r"),
                                eta=x["eta"], alpha=sl("alpha"), workspace=ws)
        os_.append(o)
        kts.append(kt)
    torch.cuda.synchronize()
    assert ws.status() == 0
    return torch.stack(kts, 2).cpu(), d.cpu(), torch.stack(os_, 2).cpu(), S.cpu()


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 20])
def test_decode_steps_match_oracle(io, T):
    for (K, V), gated in itertools.product([(64, 64), (128, 128), (128, 64)], [False, True]):
        x = synth.make_random(2, 3, T, K, V, io=io, apf=True, gated=gated, s0=True, d0=True,
                              seed=40 + T + K + V)
        gen = torch.Generator().manual_seed(7)
        d0 = x["d0"] if x["d0"] is not None else torch.ones(2, 3, K)
        S0 = x["S0"] if x["S0"] is not None else 0.1 * torch.randn(2, 3, V, K, generator=gen)
        kt, dT, o, ST = run_steps(x, d0, S0)
        okt, odT, oo, oST = oracle_steps(x, d0, S0)
        tol = TOL[io]
        errs = {"ktilde": rel_err(kt, okt), "d": rel_err(dT, odT), "o": rel_err(o, oo),
                "S": rel_err(ST, oST)}
        for name, e in errs.items():
            assert e <= tol, "%s T=%d K=%d V=%d gated=%s %s: %.3e (%s)" % (
                io, T, K, V, gated, name, e, errs)


def test_decode_step_without_optional_gates():
    # r == NULL (no retention) and alpha == NULL (no decay): d grows by the
    # plain hypergradient step, S by the plain delta rule
    x = synth.make_random(1, 4, 1, 128, 128, io="bf16", seed=9)
    d0 = torch.ones(1, 4, 128)
    S0 = torch.zeros(1, 4, 128, 128)
    kt, dT, o, ST = run_steps(x, d0, S0)
    okt, odT, oo, oST = oracle_steps(x, d0, S0)
    assert rel_err(dT, odT) <= TOL["bf16"] and rel_err(ST, oST) <= TOL["bf16"]
    assert rel_err(o, oo) <= TOL["bf16"] and rel_err(kt, okt) <= TOL["bf16"]
