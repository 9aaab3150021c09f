"""The residual diagnostic of Phase 1 (osdn_precond_scan_residual) against
the fp64 oracle: per sequence, sum_t log((1 - beta_t <d_t, k_t^2>)^2), the log
of the product of the token residual ratios of theorem 5.2 (gist.science
summary of arXiv 2605.13473, section 3), whose exp over T is the q_geo of
section 4.2.  The scan's other outputs must be those of osdn_precond_scan."""
import numpy as np
import pytest
import torch

import oracle
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


def run(x):
    g = to_cuda(x)
    ws = ops.Workspace()
    kt, dT, lr = ops.precond_scan(g["k"], g["beta"], g["r"], g["eta"], g["d0"], workspace=ws,
                                  log_ratio=True)
    kt0, dT0 = ops.precond_scan(g["k"], g["beta"], g["r"], g["eta"], g["d0"], workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    # the diagnostic changes nothing else
    assert torch.equal(kt, kt0) and torch.equal(dT, dT0)
    okt, odT, olr = oracle.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"],
                                        log_ratio=True)
    return lr, olr


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("case", ["plain", "apf_segments", "apf_tail", "eta0", "slow_retention",
                                  "expansive_token"])
def test_log_ratio_matches_oracle(io, case):
    T = {"plain": 333, "apf_segments": 3000, "apf_tail": 3001, "eta0": 200,
         "slow_retention": 3000, "expansive_token": 3000}[case]
    x = synth.make_random(2, 3, T, 128 if case != "plain" else 64, 64, io=io,
                          apf=case not in ("plain", "eta0"), d0=True, seed=40 + T)
    if case == "eta0":
        x["eta"] = 0.0
    if case == "slow_retention":      # every speculative start is repaired, with its sum
        x["r"] = torch.full_like(x["r"], 0.99995)
    if case == "expansive_token":     # every segment recomputed in the verify pass
        x["r"][:, :, 1700] = 1.5
    lr, olr = run(x)
    assert lr.shape == (2, 3)
    assert np.all(np.isfinite(olr))
    assert rel_err(lr, olr) <= TOL[io], (rel_err(lr, olr), lr, olr)


def test_log_ratio_exact_fit_and_empty():
    # beta_t <d_t, k_t^2> = 1 at one token (d = 1, unit key, beta = 1): the
    # product of ratios is 0 and the log -inf; T = 0: an empty product
    x = synth.make_random(1, 2, 40, 64, 64, io="f32", seed=5)
    x["k"][:, :, 7] = 0.0
    x["k"][:, :, 7, 3] = 1.0
    x["beta"][:, :, 7] = 1.0
    x["eta"] = 0.0                    # keeps d = 1 up to token 7
    lr, olr = run(x)
    assert np.all(np.isneginf(olr))
    assert torch.all(torch.isneginf(lr.cpu()))
    g = to_cuda(synth.make_random(1, 2, 0, 64, 64, io="bf16", seed=6))
    _, _, lr0 = ops.precond_scan(g["k"], g["beta"], g["r"], g["eta"], g["d0"], log_ratio=True)
    assert torch.equal(lr0.cpu(), torch.zeros(1, 2))
