"""The timeout path of the tensor-core Phase 2 on the GPU, without a fault:
the workspace header's test word makes the state-recurrence kernel load
nothing, so a bounded wait on a barrier that nothing completes runs out.  The call must end, leave OSDN_ERR_TIMEOUT in the
workspace status word, and leave the device usable: the same call without
the hook then matches the oracle."""
import pytest
import torch

from preconditioned_delta_rule_phase1_gb300 import build as osdn_build
from preconditioned_delta_rule_phase1_gb300 import ops, synth
from tests._util import TOL, oracle_forward, rel_err, to_cuda

pytestmark = pytest.mark.gpu

OSDN_ERR_TIMEOUT = -7


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    osdn_build.build()
    ops.lib()


@pytest.mark.parametrize("gated", [False, True])
def test_stalled_chain_reports_timeout_and_device_stays_usable(gated):
    x = synth.make_random(1, 2, 200, 64, 64, io="bf16", apf=True, gated=gated, s0=True, seed=71)
    g = to_cuda(x)
    kt, dT = ops.precond_scan(g["k"], g["beta"], g["r"], g["eta"], g["d0"])
    ws = ops.Workspace()
    ws.ensure(ops.chunk_fwd_workspace_bytes(1, 1, 2, 200, 64, 64))
    ws.buf[4:8].view(torch.int32).fill_(1)    # the header's test word
    ops.chunk_fwd(g["q"], g["k"], kt, g["v"], g["beta"], g["alpha"], g["S0"], workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == OSDN_ERR_TIMEOUT
    ws2 = ops.Workspace()
    o, ST = ops.chunk_fwd(g["q"], g["k"], kt, g["v"], g["beta"], g["alpha"], g["S0"], workspace=ws2)
    torch.cuda.synchronize()
    assert ws2.status() == 0
    _, _, oo, oST = oracle_forward(x)
    assert rel_err(o, oo) <= TOL["bf16"]
    assert rel_err(ST, oST) <= TOL["bf16"]
