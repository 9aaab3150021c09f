"""The library's calls inside CUDA graphs.

A caller that replays a fixed step many times (serving, a training loop) can
capture the calls into a CUDA graph once and replay it, instead of paying
the launches every step.  The multi-slab bf16 Phase 2 forks onto two
library-owned streams and joins back with events; under capture those
streams join the caller's capture, so the whole schedule becomes part of the
graph.  Each case captures after one eager warm-up call (which sets the
kernels' shared-memory attributes and creates the library's streams),
replays the graph on fresh inputs copied into the captured buffers, and
requires the replay to equal an eager call on the same inputs bit for bit.
"""
import pytest
import torch

from preconditioned_delta_rule_phase1_gb300 import build as osdn_build
from preconditioned_delta_rule_phase1_gb300 import ops, synth
from tests._util import to_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    osdn_build.build()
    ops.lib()


def captured(fn, bufs, fresh):
    """Warm up, capture fn() into a graph, copy `fresh` into `bufs`, replay."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = fn()
    for name, t in fresh.items():
        bufs[name].copy_(t)
    g.replay()
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("T,gated", [(64 * 130 + 5, False), (64 * 48, True), (300, True)])
def test_two_call_forward_in_a_graph(T, gated):
    # 131 chunks: three slabs on the library's streams; 48 chunks with a
    # decay: the time-segmented chain; 300 tokens: one slab
    a = to_cuda(synth.make_random(1, 2, T, 128, 128, io="bf16", apf=True, gated=gated, s0=True,
                                  d0=True, seed=T))
    b = to_cuda(synth.make_random(1, 2, T, 128, 128, io="bf16", apf=True, gated=gated, s0=True,
                                  d0=True, seed=T + 1))
    ws = ops.Workspace()
    ws.ensure(max(ops.precond_scan_workspace_bytes(1, 2, T, 128),
                  ops.chunk_fwd_workspace_bytes(1, 1, 2, T, 128, 128)))
    fn = lambda: ops.forward(a["q"], a["k"], a["v"], a["beta"], a["r"], a["eta"], a["d0"],
                             a["alpha"], a["S0"], workspace=ws)
    names = [n for n in ("q", "k", "v", "beta", "r", "d0", "alpha", "S0") if a[n] is not None]
    got = captured(fn, a, {n: b[n] for n in names})
    assert ws.status() == 0
    ref = ops.forward(b["q"], b["k"], b["v"], b["beta"], b["r"], b["eta"], b["d0"], b["alpha"],
                      b["S0"])
    torch.cuda.synchronize()
    for x, y in zip(got, ref):
        assert torch.equal(x, y)


def test_one_call_forward_in_a_graph():
    T = 64 * 70 + 9
    a = to_cuda(synth.make_random(1, 2, T, 128, 64, io="bf16", apf=True, s0=True, seed=7))
    b = to_cuda(synth.make_random(1, 2, T, 128, 64, io="bf16", apf=True, s0=True, seed=8))
    ws = ops.Workspace()
    ws.ensure(ops.forward_workspace_bytes(1, 1, 2, T, 128, 64))
    fn = lambda: ops.forward_fused(a["q"], a["k"], a["v"], a["beta"], a["r"], a["eta"], None,
                                   None, a["S0"], workspace=ws)
    got = captured(fn, a, {n: b[n] for n in ("q", "k", "v", "beta", "r", "S0")})
    assert ws.status() == 0
    ref = ops.forward_fused(b["q"], b["k"], b["v"], b["beta"], b["r"], b["eta"], None, None,
                            b["S0"])
    torch.cuda.synchronize()
    for x, y in zip(got, ref):
        assert torch.equal(x, y)


def test_decode_steps_in_a_graph():
    # eight chained decode steps captured once; the state updates in place
    B, H, K, V, n = 4, 4, 128, 128, 8
    x = to_cuda(synth.make_random(B, H, n, K, V, io="bf16", apf=True, gated=True, seed=9))
    d = torch.ones(B, H, K, device="cuda")
    S = torch.zeros(B, H, V, K, device="cuda")
    tok = {name: x[name][:, :, 0].contiguous() for name in ("q", "k", "v", "beta", "r", "alpha")}
    ws = ops.Workspace()
    o = torch.empty(B, H, V, dtype=torch.bfloat16, device="cuda")
    kt = torch.empty(B, H, K, dtype=torch.bfloat16, device="cuda")

    def fn():
        for _ in range(n):
            ops.decode_step(tok["q"], tok["k"], tok["v"], tok["beta"], d, S, tok["r"], x["eta"],
                            tok["alpha"], o, kt, ws)
        return o
    # warm-up and capture advance the state; start both paths from the same one
    captured(fn, {}, {})
    d0, S0 = d.clone(), S.clone()
    torch.cuda.synchronize()
    d.copy_(d0)
    S.copy_(S0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    d.copy_(d0)
    S.copy_(S0)
    g.replay()
    torch.cuda.synchronize()
    got_d, got_S, got_o = d.clone(), S.clone(), o.clone()
    d.copy_(d0)
    S.copy_(S0)
    fn()
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert torch.equal(got_d, d) and torch.equal(got_S, S) and torch.equal(got_o, o)


def test_backward_in_a_graph():
    # the three backward kernels and the checkpoint scan, replayed on fresh
    # inputs and cotangents, against an eager call on the same inputs
    B, H, T, K, V = 1, 2, 300, 128, 64
    xs = []
    for seed in (21, 22):
        x = to_cuda(synth.make_random(B, H, T, K, V, io="bf16", apf=True, gated=True, s0=True,
                                      d0=True, seed=seed))
        x["kt"], _ = ops.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"])
        gen = torch.Generator().manual_seed(seed)
        x["do"] = torch.randn(B, H, T, V, generator=gen).to(torch.bfloat16).cuda()
        xs.append(x)
    a, b = xs
    ws = ops.Workspace()
    ws.ensure(ops.backward_workspace_bytes(B, H, T, K, V))
    fn = lambda: ops.backward(a["q"], a["k"], a["kt"], a["v"], a["beta"], a["r"], a["eta"],
                              a["d0"], a["alpha"], a["S0"], do=a["do"], workspace=ws)
    names = ("q", "k", "kt", "v", "beta", "r", "d0", "alpha", "S0", "do")
    got = captured(fn, a, {n: b[n] for n in names})
    assert ws.status() == 0
    ref = ops.backward(b["q"], b["k"], b["kt"], b["v"], b["beta"], b["r"], b["eta"], b["d0"],
                       b["alpha"], b["S0"], do=b["do"])
    torch.cuda.synchronize()
    assert set(got) == set(ref)
    for n in ref:
        assert torch.equal(got[n], ref[n]), n


def test_per_channel_decay_forward_in_a_graph():
    # the tensor-core Phase 2 with a decay per key channel over several slabs
    B, H, T, K, V = 1, 2, 64 * 70 + 9, 128, 128
    xs = []
    for seed in (23, 24):
        x = to_cuda(synth.make_random(B, H, T, K, V, io="bf16", apf=True, s0=True, d0=True,
                                      seed=seed))
        gen = torch.Generator().manual_seed(seed)
        x["ak"] = (0.9 + 0.1 * torch.rand(B, H, T, K, generator=gen)).cuda()
        xs.append(x)
    a, b = xs
    ws = ops.Workspace()
    fn = lambda: ops.forward_kda(a["q"], a["k"], a["v"], a["beta"], a["r"], a["eta"], a["d0"],
                                 a["ak"], a["S0"], workspace=ws)
    names = ("q", "k", "v", "beta", "r", "d0", "ak", "S0")
    got = captured(fn, a, {n: b[n] for n in names})
    assert ws.status() == 0
    ref = ops.forward_kda(b["q"], b["k"], b["v"], b["beta"], b["r"], b["eta"], b["d0"], b["ak"],
                         b["S0"])
    torch.cuda.synchronize()
    for x, y in zip(got, ref):
        assert torch.equal(x, y)
