"""The Python binding's argument checks, on the CPU with a stand-in library.

The C ABI takes plain pointers, so the binding checks every tensor's shape,
dtype and device before a pointer leaves Python (a wrong-sized tensor would
otherwise be read or written out of its bounds).  Here the library is a fake
that records calls and the device context is a no-op, so the checks run on
CPU tensors: every call pattern the GPU tests use must pass them, and each
kind of mistake must be refused before the library is called.
"""
import contextlib
import ctypes

import pytest
import torch

from preconditioned_delta_rule_phase1_gb300 import ops, synth


class FakeLib:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if not name.startswith("osdn_"):
            raise AttributeError(name)

        def fn(*args):
            self.calls.append(name)
            return 256 if name.endswith("workspace_bytes") else 0
        return fn


@pytest.fixture
def fake(monkeypatch):
    lib = FakeLib()
    monkeypatch.setattr(ops, "lib", lambda: lib)
    monkeypatch.setattr(ops, "_on", lambda device: contextlib.nullcontext())
    monkeypatch.setattr(ops, "_stream", lambda stream, device=None: ctypes.c_void_p(0))
    monkeypatch.setattr(ops, "_ptr", lambda t: None if t is None else ctypes.c_void_p(1))
    return lib


def inputs(io="bf16", K=64, V=64, **kw):
    return synth.make_random(2, 3, 40, K, V, io=io, **kw)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [{}, dict(apf=True, gated=True, s0=True, d0=True)])
def test_valid_calls_pass(fake, io, opts):
    x = inputs(io, K=128, V=64, **opts)
    kt, dT = ops.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"])
    kt, dT, lr = ops.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"], log_ratio=True)
    assert lr.shape == (2, 3)
    ops.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"], kt, dT, ops.Workspace(device="cpu"))
    ops.precond_scan_noalloc(x["k"], x["beta"], x["r"], x["eta"], x["d0"])
    o, ST = ops.chunk_fwd(x["q"], x["k"], kt, x["v"], x["beta"], x["alpha"], x["S0"],
                          workspace=ops.Workspace(device="cpu"))
    assert o.shape == (2, 3, 40, 64) and ST.shape == (2, 3, 64, 128)
    ops.forward(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"], x["alpha"], x["S0"],
                workspace=ops.Workspace(device="cpu"))
    d = torch.ones(2, 3, 128)
    S = torch.zeros(2, 3, 64, 128)
    sl = lambda n: None if x[n] is None else x[n][:, :, 0].contiguous()
    ops.decode_step(sl("q"), sl("k"), sl("v"), sl("beta"), d, S, r=sl("r"), eta=x["eta"],
                    alpha=sl("alpha"), workspace=ops.Workspace(device="cpu"))
    g = ops.backward(x["q"], x["k"], kt, x["v"], x["beta"], x["r"], x["eta"], x["d0"], x["alpha"],
                     x["S0"], do=torch.zeros(2, 3, 40, 64, dtype=x["k"].dtype),
                     dST=torch.zeros(2, 3, 64, 128), ddT=torch.zeros(2, 3, 128),
                     dktilde=torch.zeros_like(kt), workspace=ops.Workspace(device="cpu"))
    want = {"q", "k", "v", "beta", "eta"} | {n for n in ("r", "alpha", "d0", "S0")
                                             if x[n] is not None}
    assert set(g) == want and g["eta"].shape == (2, 3) and g["S0" if "S0" in g else "q"].numel()
    assert "osdn_decode_step" in fake.calls and "osdn_precond_scan_residual" in fake.calls
    assert "osdn_backward" in fake.calls
    ak = torch.rand(2, 3, 40, 128)
    o, ST = ops.chunk_fwd_kda(x["q"], x["k"], kt, x["v"], x["beta"], ak, x["S0"],
                              workspace=ops.Workspace(device="cpu"))
    assert o.shape == (2, 3, 40, 64) and ST.shape == (2, 3, 64, 128)
    ops.forward_kda(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"], ak, x["S0"],
                    workspace=ops.Workspace(device="cpu"))
    gk = ops.backward_kda(x["q"], x["k"], kt, x["v"], x["beta"], x["r"], x["eta"], x["d0"], ak,
                          x["S0"], do=torch.zeros(2, 3, 40, 64, dtype=x["k"].dtype),
                          workspace=ops.Workspace(device="cpu"))
    assert gk["alpha"].shape == (2, 3, 40, 128)
    ops.decode_step_kda(sl("q"), sl("k"), sl("v"), sl("beta"), d, S, r=sl("r"), eta=x["eta"],
                        alpha_k=ak[:, :, 0].contiguous(), workspace=ops.Workspace(device="cpu"))
    assert "osdn_chunk_fwd_kda" in fake.calls and "osdn_backward_kda" in fake.calls
    assert "osdn_decode_step_kda" in fake.calls


def test_mistakes_are_refused_before_the_library(fake):
    x = inputs("bf16", apf=True, gated=True, s0=True, d0=True)
    ws = ops.Workspace(device="cpu")
    bad = [
        lambda: ops.precond_scan(x["k"], x["beta"].bfloat16(), x["r"]),             # beta dtype
        lambda: ops.precond_scan(x["k"], x["beta"][:, :, :-1], x["r"]),              # beta length
        lambda: ops.precond_scan(x["k"], x["beta"], x["r"], d0=x["d0"][..., :32]),   # d0 width
        lambda: ops.precond_scan(x["k"], x["beta"], ktilde=torch.empty(2, 3, 40, 64)),  # ktilde dtype
        lambda: ops.precond_scan(x["k"], x["beta"], log_ratio=torch.empty(3, 2)),    # log_ratio shape
        lambda: ops.chunk_fwd(x["q"], x["k"], x["k"], x["v"][:, :, :20], x["beta"]),  # v length
        lambda: ops.chunk_fwd(x["q"].float(), x["k"], x["k"], x["v"], x["beta"]),     # q dtype
        lambda: ops.chunk_fwd(x["q"], x["k"], x["k"], x["v"], x["beta"],
                              S0=x["S0"].transpose(-1, -2)),                          # S0 layout
        lambda: ops.chunk_fwd(x["q"], x["k"], x["k"], x["v"], x["beta"], x["alpha"][0]),  # alpha
        lambda: ops.decode_step(x["q"][:, :, 0], x["k"][:, :, 0], x["v"][:, :, 0],
                                x["beta"], torch.ones(2, 3, 64),
                                torch.zeros(2, 3, 64, 64), workspace=ws),             # beta per token
        lambda: ops.decode_step(x["q"][:, :, 0], x["k"][:, :, 0], x["v"][:, :, 0],
                                x["beta"][:, :, 0], torch.ones(2, 3, 64).double(),
                                torch.zeros(2, 3, 64, 64), workspace=ws),             # d dtype
        lambda: ops.backward(x["q"], x["k"], x["k"], x["v"], x["beta"],
                             do=x["v"].float(), workspace=ws),                       # do dtype
        lambda: ops.backward(x["q"], x["k"], x["k"], x["v"], x["beta"],
                             dST=torch.zeros(2, 3, 64, 32), workspace=ws),           # dST shape
        lambda: ops.backward(x["q"], x["k"], None, x["v"], x["beta"], workspace=ws),  # no ktilde
        lambda: ops.chunk_fwd_kda(x["q"], x["k"], x["k"], x["v"], x["beta"], x["alpha"],
                                  workspace=ws),                        # a scalar gate for KDA
        lambda: ops.backward_kda(x["q"], x["k"], x["k"], x["v"], x["beta"],
                                 alpha_k=x["alpha"], workspace=ws),     # likewise
        lambda: ops.backward(x["q"], x["k"], x["k"], x["v"], x["beta"],
                             alpha=torch.rand(2, 3, 40, 64), workspace=ws),  # per-channel gate
    ]
    for i, call in enumerate(bad):
        n = len(fake.calls)
        with pytest.raises((ValueError, TypeError)):
            call()
        assert not [c for c in fake.calls[n:] if not c.endswith("workspace_bytes")], i


def test_cpu_tensors_are_refused_without_the_fake():
    # with the real device context, CPU tensors never reach the library
    x = inputs("f32")
    with pytest.raises(ValueError):
        ops.precond_scan(x["k"], x["beta"], workspace=ops.Workspace(device="cpu"))
