"""osdn_precond_scan_noalloc: the Phase 1 scan for callers that cannot call
cudaMalloc (a capture region whose memory pool forbids new allocations, a
host framework that owns every allocation, a service that must not meet
out-of-memory after start-up).  Its scratch is a static device array inside
the library, so it needs no workspace argument.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It must pass both alone in
a fresh process and after the other tests (the static scratch then holds the
contents of earlier calls).
"""
import ctypes

import pytest
import torch

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


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    # two different problems back to back through the static scratch; both
    # use speculative segments (retention gate given), so the scratch is used
    cases = [
        dict(B=2, H=16, T=8192, K=128, io="bf16", seed=31),
        dict(B=1, H=6, T=5000, K=64, io="f32", seed=32),
    ]
    for c in cases:
        x = to_cuda(synth.make_random(c["B"], c["H"], c["T"], c["K"], 64, io=c["io"], apf=True,
                                      d0=True, seed=c["seed"]))
        ws = ops.Workspace()
        kt_ref, dT_ref = ops.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"],
                                          workspace=ws)
        kt, dT = ops.precond_scan_noalloc(x["k"], x["beta"], x["r"], x["eta"], x["d0"])
        torch.cuda.synchronize()
        assert ws.status() == 0
        tol = TOL[c["io"]]
        assert rel_err(kt, kt_ref.double().cpu().numpy()) <= tol
        assert rel_err(dT, dT_ref.double().cpu().numpy()) <= tol


def test_noalloc_rejects_shapes_beyond_its_scratch():
    L = ops.lib()
    # fake, widely spaced addresses: the size check fails before any is used
    k, beta, r, kt = (ctypes.c_void_p(i << 40) for i in (1, 2, 3, 4))
    code = L.osdn_precond_scan_noalloc(1, 1, 512, 65536, 128, k, beta, r, 0.1, None, kt, None,
                                       None)
    assert code == -11, ops.status_string(code)
