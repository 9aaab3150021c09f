"""osdn_precond_scan_noalloc: the Phase 1 scan for callers that cannot call
cudaMalloc (a capture region whose memory pool forbids new allocations, a
host framework that owns every allocation, a service that must not meet
out-of-memory after start-up).  Its scratch is a static device array inside
the library, so it needs no workspace argument.

The allocation-free call runs the same kernels as osdn_precond_scan, so the
two must agree bit for bit; a scratch-layout slip or stale scratch contents
would show up here even where the scan's verify step would repair them.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It must pass both alone in
a fresh process and after the other tests (the static scratch then holds the
contents of earlier calls).
"""
import pytest
import torch

from preconditioned_delta_rule_phase1_gb300 import build as osdn_build
from preconditioned_delta_rule_phase1_gb300 import ops, synth
from tests._util import TOL, pick, rel_err, to_cuda

pytestmark = pytest.mark.gpu

OSDN_ERR_SCRATCH = -11


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    osdn_build.build()
    ops.lib()


def both(x):
    ws = ops.Workspace()
    kt_ref, dT_ref = ops.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"], workspace=ws)
    kt, dT = ops.precond_scan_noalloc(x["k"], x["beta"], x["r"], x["eta"], x["d0"])
    torch.cuda.synchronize()
    assert ws.status() == 0
    return kt, dT, kt_ref, dT_ref


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    # the largest case first, so that the smaller ones after it find the static
    # scratch full of another problem's segment states; every case but the
    # ungated and the empty one uses speculative segments (a retention gate)
    cases = [
        dict(B=2, H=16, T=8192, K=128, io="bf16", apf=True, seed=31),
        dict(B=1, H=6, T=5000, K=64, io="f32", apf=True, seed=32),
        dict(B=1, H=6, T=5000, K=64, io="f32", apf=True, seed=33),
        dict(B=2, H=3, T=700, K=128, io="bf16", apf=False, seed=34),
        dict(B=1, H=2, T=0, K=64, io="f32", apf=True, seed=35),
    ]
    import oracle
    for c in cases:
        x = synth.make_random(c["B"], c["H"], c["T"], c["K"], 64, io=c["io"], apf=c["apf"],
                              d0=True, seed=c["seed"])
        g = to_cuda(x)
        kt, dT, kt_ref, dT_ref = both(g)
        assert torch.equal(kt, kt_ref), c
        assert torch.equal(dT, dT_ref), c
        # and against the oracle, on the first and the last sequence
        if c["T"] > 0:
            heads = sorted({0, c["B"] * c["H"] - 1})
            xs = synth.slice_heads(x, heads)
            okt, odT = oracle.precond_scan(xs["k"], xs["beta"], xs["r"], xs["eta"], xs["d0"])
            assert rel_err(pick(kt, heads), okt) <= TOL[c["io"]], c
            assert rel_err(pick(dT, heads), odT) <= TOL[c["io"]], c


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 2048 sequences of 1025 tokens with a retention gate: two speculative
    # segments a sequence, about 4 MB of segment states, twice the static
    # array.  Real tensors (about 0.5 GB of keys), so that no check order could
    # ever hand a kernel an address that is not a live allocation.
    B, H, T, K = 16, 128, 1025, 128
    k = torch.zeros(B, H, T, K, dtype=torch.bfloat16, device="cuda")
    beta = torch.full((B, H, T), 0.5, device="cuda")
    r = torch.full((B, H, T), 0.9, device="cuda")
    kt = torch.empty_like(k)
    L = ops.lib()
    code = L.osdn_precond_scan_noalloc(1, B, H, T, K, ops._ptr(k), ops._ptr(beta), ops._ptr(r),
                                       0.1, None, ops._ptr(kt), None, None)
    assert code == OSDN_ERR_SCRATCH, ops.status_string(code)
    # a smaller batch of the same length fits the static array and runs
    code = L.osdn_precond_scan_noalloc(1, 1, 64, T, K, ops._ptr(k), ops._ptr(beta), ops._ptr(r),
                                       0.1, None, ops._ptr(kt), None, None)
    torch.cuda.synchronize()
    assert code == 0, ops.status_string(code)


def test_noalloc_in_a_graph_with_preallocated_outputs():
    # the use the entry point exists for: a capture into which nothing is
    # allocated (outputs given), replayed on fresh keys and gates, equal to
    # an eager call bit for bit
    B, H, T, K = 2, 8, 3000, 128
    xs = [to_cuda(synth.make_random(B, H, T, K, 64, io="bf16", apf=True, d0=True, seed=s))
          for s in (41, 42)]
    a, b = xs
    kt = torch.empty_like(a["k"])
    dT = torch.empty(B, H, K, device="cuda")
    fn = lambda: ops.precond_scan_noalloc(a["k"], a["beta"], a["r"], a["eta"], a["d0"], kt, dT)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()   # sets the kernels' attributes outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for n in ("k", "beta", "r", "d0"):
        a[n].copy_(b[n])
    g.replay()
    torch.cuda.synchronize()
    kt_ref, dT_ref = ops.precond_scan_noalloc(b["k"], b["beta"], b["r"], b["eta"], b["d0"])
    torch.cuda.synchronize()
    assert torch.equal(kt, kt_ref) and torch.equal(dT, dT_ref)
