"""The per-channel decay (osdn_chunk_fwd_kda, osdn_backward_kda) against the
fp64 oracle: Phase 2 with S_t = S_{t-1} Diag(alpha_t) + beta_t (v_t - S_{t-1}
Diag(alpha_t) k_t) ktilde_t^T (the Kimi-Delta-Attention-style reading of the
backbone named in section 4 of the gist.science summary), both phases through
the C ABI against ``oracle.forward_kda``, and the gradients against the
autograd reference with a per-channel alpha.  Normwise tolerances of the I/O
type; both I/O types, every (K, V), ragged token counts, T = 0, no decay,
equal channels against the scalar-gate call, determinism.  bf16 runs on the
tensor cores (the decay folded into the chunk operands per channel against
a reference point per 16-token block): long sequences cut into slabs and
into time segments, decays down to the supported 2^-6, and a decay outside
the supported range reported in the status word.
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


def decay(B, H, T, K, seed, low=0.6):
    g = torch.Generator().manual_seed(seed)
    return (low + (1 - low) * torch.rand(B, H, T, K, generator=g)).contiguous()


def case(io, K, V, T, seed):
    x = synth.make_random(1, 2, T, K, V, io=io, apf=True, s0=True, d0=True, seed=seed)
    x["alpha"] = decay(1, 2, T, K, seed + 1)
    return x


FWD = [("f32", 64, 64, 37), ("f32", 128, 128, 100), ("f32", 128, 64, 1),
       ("bf16", 128, 128, 100), ("bf16", 64, 128, 33), ("bf16", 64, 64, 16)]


@pytest.mark.parametrize("io,K,V,T", FWD)
def test_forward_matches_oracle(io, K, V, T):
    x = case(io, K, V, T, 300 + T + K)
    g = to_cuda(x)
    got = ops.forward_kda(g["q"], g["k"], g["v"], g["beta"], g["r"], g["eta"], g["d0"],
                          g["alpha"], g["S0"])
    torch.cuda.synchronize()
    ref = oracle.forward_kda(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"],
                             x["alpha"], x["S0"])
    errs = {n: rel_err(a, b) for n, a, b in zip(("ktilde", "dT", "o", "ST"), got, ref)}
    assert max(errs.values()) <= TOL[io], errs


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_no_decay_and_empty(io):
    x = case(io, 64, 64, 40, 11)
    g = to_cuda(x)
    kt, _ = ops.precond_scan(g["k"], g["beta"], g["r"], g["eta"], g["d0"])
    o, ST = ops.chunk_fwd_kda(g["q"], g["k"], kt, g["v"], g["beta"], None, g["S0"])
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.delta_fwd(x["q"], x["k"], kt.cpu(), x["v"], x["beta"], None, x["S0"])
    assert rel_err(o, o_ref) <= TOL[io] and rel_err(ST, S_ref) <= TOL[io]
    e = case(io, 64, 64, 0, 12)
    ge = to_cuda(e)
    o0, S0 = ops.chunk_fwd_kda(ge["q"], ge["k"], ge["k"], ge["v"], ge["beta"], ge["alpha"],
                               ge["S0"])
    torch.cuda.synchronize()
    assert o0.numel() == 0 and torch.equal(S0.cpu(), e["S0"])


def test_equal_channels_match_the_scalar_gate():
    x = synth.make_random(1, 2, 70, 128, 64, io="f32", apf=True, gated=True, s0=True, seed=13)
    g = to_cuda(x)
    kt, _ = ops.precond_scan(g["k"], g["beta"], g["r"], g["eta"])
    ak = g["alpha"][..., None].expand(1, 2, 70, 128).contiguous()
    o1, S1 = ops.chunk_fwd(g["q"], g["k"], kt, g["v"], g["beta"], g["alpha"], g["S0"])
    o2, S2 = ops.chunk_fwd_kda(g["q"], g["k"], kt, g["v"], g["beta"], ak, g["S0"])
    torch.cuda.synchronize()
    # the two kernels round differently (decay before or after the dot
    # product), so they agree to the fp32 tolerance, not bit for bit
    assert rel_err(o2, o1.double().cpu().numpy()) <= TOL["f32"]
    assert rel_err(S2, S1.double().cpu().numpy()) <= TOL["f32"]


@pytest.mark.parametrize("K,V,T,low,high", [
    (128, 128, 64 * 130 + 17, 0.6, 1.0),     # slabs of chunks, a ragged last chunk
    (64, 64, 64 * 48, 0.9, 1.0),             # a time-segmented chain (3 segments)
    (128, 64, 64 * 48, 0.999, 1.0),          # ... whose speculative starts are repaired
    (128, 128, 300, 0.015625, 0.2),          # decays down to 2^-6: reference points matter
    (64, 128, 150, 1.0, 1.0),                # alpha = 1 everywhere
])
def test_bf16_tensor_core_path(K, V, T, low, high):
    x = synth.make_random(1, 2, T, K, V, io="bf16", apf=True, s0=True, d0=True, seed=T + K)
    g = torch.Generator().manual_seed(T + V)
    x["alpha"] = (low + (high - low) * torch.rand(1, 2, T, K, generator=g)).contiguous()
    gx = to_cuda(x)
    ws = ops.Workspace()
    got = ops.forward_kda(gx["q"], gx["k"], gx["v"], gx["beta"], gx["r"], gx["eta"], gx["d0"],
                          gx["alpha"], gx["S0"], workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0, ops.status_string(ws.status())
    ref = oracle.forward_kda(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"],
                             x["alpha"], x["S0"])
    errs = {n: rel_err(a, b) for n, a, b in zip(("ktilde", "dT", "o", "ST"), got, ref)}
    assert max(errs.values()) <= TOL["bf16"], errs
    # Phase 2 alone from the GPU's own ktilde
    o2, S2 = oracle.delta_fwd_kda(x["q"], x["k"], got[0].cpu(), x["v"], x["beta"], x["alpha"],
                                  x["S0"])
    assert rel_err(got[2], o2) <= TOL["bf16"] and rel_err(got[3], S2) <= TOL["bf16"]


@pytest.mark.parametrize("bad", [0.0, 0.01, 100.0, float("nan")])
def test_bf16_decay_outside_the_supported_range_is_reported(bad):
    x = case("bf16", 64, 64, 100, 17)
    g = to_cuda(x)
    g["alpha"][0, 1, 70, 5] = bad
    kt, _ = ops.precond_scan(g["k"], g["beta"], g["r"], g["eta"], g["d0"])
    ws = ops.Workspace()
    ops.chunk_fwd_kda(g["q"], g["k"], kt, g["v"], g["beta"], g["alpha"], g["S0"], workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == -8, ops.status_string(ws.status())
    # the same inputs in fp32 run the FFMA recurrence, which takes any decay
    ok = ops.Workspace()
    ops.chunk_fwd_kda(g["q"].float(), g["k"].float(), kt.float(), g["v"].float(), g["beta"],
                      g["alpha"].nan_to_num(0.5), g["S0"], workspace=ok)
    torch.cuda.synchronize()
    assert ok.status() == 0


def test_bf16_equal_channels_match_the_scalar_gate():
    x = synth.make_random(1, 2, 700, 128, 128, io="bf16", apf=True, gated=True, s0=True, seed=19)
    g = to_cuda(x)
    kt, _ = ops.precond_scan(g["k"], g["beta"], g["r"], g["eta"])
    ak = g["alpha"][..., None].expand(1, 2, 700, 128).contiguous()
    o1, S1 = ops.chunk_fwd(g["q"], g["k"], kt, g["v"], g["beta"], g["alpha"], g["S0"])
    o2, S2 = ops.chunk_fwd_kda(g["q"], g["k"], kt, g["v"], g["beta"], ak, g["S0"])
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.delta_fwd(x["q"], x["k"], kt.cpu(), x["v"], x["beta"], x["alpha"],
                                    x["S0"])
    for a, b in ((o1, o_ref), (o2, o_ref), (S1, S_ref), (S2, S_ref)):
        assert rel_err(a, b) <= TOL["bf16"]


def test_bf16_deterministic():
    x = case("bf16", 128, 128, 1000, 23)
    g = to_cuda(x)
    a = ops.forward_kda(g["q"], g["k"], g["v"], g["beta"], g["r"], g["eta"], g["d0"], g["alpha"],
                        g["S0"])
    b = ops.forward_kda(g["q"], g["k"], g["v"], g["beta"], g["r"], g["eta"], g["d0"], g["alpha"],
                        g["S0"])
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v)


BWD = [("f32", 64, 64, 50), ("f32", 128, 64, 5), ("bf16", 128, 128, 100), ("bf16", 64, 128, 33)]


def stored_ktilde(x):
    kt, _ = oracle.precond_scan(x["k"], x["beta"], x["r"], x["eta"], x["d0"])
    return torch.from_numpy(np.asarray(kt)).to(x["k"].dtype).contiguous()


def run_backward(x, cot, kt):
    g, c = to_cuda(x), to_cuda(cot)
    got = ops.backward_kda(g["q"], g["k"], kt.cuda(), g["v"], g["beta"], g["r"], g["eta"],
                           g["d0"], g["alpha"], g["S0"], do=c["o"], dST=c["ST"], ddT=c["dT"],
                           dktilde=c["kt"])
    torch.cuda.synchronize()
    return got


def cotangents(x, io, seed):
    B, H, T, K = x["k"].shape
    V = x["v"].shape[-1]
    gen = torch.Generator().manual_seed(seed)
    dt = synth.torch_dtype(io)
    return {"o": torch.randn(B, H, T, V, generator=gen).to(dt),
            "ST": torch.randn(B, H, V, K, generator=gen),
            "dT": torch.randn(B, H, K, generator=gen),
            "kt": torch.randn(B, H, T, K, generator=gen).to(dt)}


@pytest.mark.parametrize("io,K,V,T", BWD)
def test_backward_matches_reference(io, K, V, T):
    x = case(io, K, V, T, 600 + T + K)
    cot = cotangents(x, io, 700 + T)
    kt = stored_ktilde(x)
    got = run_backward(x, cot, kt)
    ref = backward.grads(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"],
                         x["alpha"], x["S0"], do=cot["o"], ddT=cot["dT"], dST=cot["ST"],
                         dkt=cot["kt"], ktilde=kt)
    assert set(got) == set(ref)
    errs = {}
    for n, r in ref.items():
        val = torch.tensor(got[n].double().sum().item()) if n == "eta" else got[n]
        errs[n] = rel_err(val, np.asarray(r))
    assert got["alpha"].shape == x["alpha"].shape
    assert max(errs.values()) <= TOL[io], errs


def test_backward_deterministic():
    x = case("bf16", 128, 64, 45, 81)
    cot = cotangents(x, "bf16", 82)
    kt = stored_ktilde(x)
    a, b = run_backward(x, cot, kt), run_backward(x, cot, kt)
    for n in a:
        assert torch.equal(a[n], b[n]), n


@pytest.mark.parametrize("io,K,V", [("f32", 64, 128), ("bf16", 128, 128), ("bf16", 64, 64)])
def test_decode_steps_match_oracle(io, K, V):
    # twenty chained per-channel decode steps against the oracle's 20-token forward
    x = case(io, K, V, 20, 900 + K + V)
    d = x["d0"].clone().cuda()
    S = x["S0"].clone().cuda()
    g = to_cuda(x)
    outs, kts = [], []
    for t in range(20):
        sl = lambda n: g[n][:, :, t].contiguous()
        o, kt = ops.decode_step_kda(sl("q"), sl("k"), sl("v"), sl("beta"), d, S, r=sl("r"),
                                    eta=x["eta"], alpha_k=sl("alpha"))
        outs.append(o)
        kts.append(kt)
    torch.cuda.synchronize()
    kt_ref, dT_ref, o_ref, S_ref = oracle.forward_kda(x["q"], x["k"], x["v"], x["beta"], x["r"],
                                                      x["eta"], x["d0"], x["alpha"], x["S0"])
    errs = {"o": rel_err(torch.stack(outs, 2), o_ref), "ktilde": rel_err(torch.stack(kts, 2), kt_ref),
            "d": rel_err(d, dT_ref), "S": rel_err(S, S_ref)}
    assert max(errs.values()) <= TOL[io], errs
