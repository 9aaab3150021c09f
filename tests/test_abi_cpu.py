"""The C-ABI library loads, exports every symbol include/osdn.h declares, and
rejects bad arguments on the host before touching the device.  No compute
call runs here (no GPU needed)."""
import ctypes
import os
import re

import pytest

from preconditioned_delta_rule_phase1_gb300 import build as osdn_build
from preconditioned_delta_rule_phase1_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    osdn_build.build()
    return ops.lib()


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(osdn_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(L):
    names = declared_functions()
    assert "osdn_precond_scan" in names and "osdn_chunk_fwd" in names
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    assert ops.status_string(0) == "ok"
    for code in range(-1, -11, -1):
        s = ops.status_string(code)
        assert s and s != "unknown status", code
    assert ops.status_string(12345) == "unknown status"
    assert L.osdn_version() >= 100


def test_workspace_sizes(L):
    assert ops.precond_scan_workspace_bytes(2, 16, 8192, 128) >= 256
    assert ops.chunk_fwd_workspace_bytes(1, 2, 16, 8192, 128, 128) >= 256


@pytest.mark.parametrize("B,H,T,K", [(2, 16, 8192, 128), (1, 16, 65536, 128), (4, 16, 4096, 64),
                                     (8, 8, 2048, 128), (1, 6, 5000, 64), (64, 32, 8192, 128),
                                     (1, 1, 257, 64), (1, 2, 256, 64)])
def test_bench_segment_rule_matches_the_library(L, B, H, T, K):
    # bench.py counts launches from a copy of the library's segment rule; the
    # library's Phase 1 workspace holds, per segment, its start and end state
    # (8 K bytes) and two 4-byte words, each array padded to 256 bytes
    import bench
    nseg = bench.precond_segments(B * H, T, True)
    n = B * H * nseg
    pad = lambda x: (x + 255) // 256 * 256
    want = 256 + (n * K * 8 + 2 * pad(n * 4) if nseg > 1 else 0)
    assert ops.precond_scan_workspace_bytes(B, H, T, K) == want


def test_bench_launch_count_rule():
    # bench.py's gpu_launches claim, from a copy of the library's schedule at
    # 152 SMs; the ncu launch lists of the 1.3B and long gated workloads show
    # 6 and 7 of the library's kernels per step
    import bench
    from preconditioned_delta_rule_phase1_gb300 import synth
    want = {"tiny_f32": 2, "lm340m_bf16": 3, "recall_apf_bf16": 6, "lm1p3b_apf_bf16": 6,
            "long_gated_apf_bf16": 7}
    for name, n in want.items():
        w = synth.WORKLOADS[name]
        x = {"r": 1 if w.apf else None, "alpha": 1 if w.gated else None}
        assert bench.launches_per_step(w, x, sms=152) == n, name
    # a per-channel decay at the 1.3B shape: the scan (2), one preparation
    # launch and a chain in two time segments (speculative pass + 1 repair)
    w = synth.WORKLOADS["lm1p3b_apf_bf16"]
    assert bench.launches_per_step(w, {"r": 1, "alpha": None}, per_channel=True, sms=152) == 5
    # the backward at that shape: checkpoint scan (2), the state adjoint's
    # forward sweep, its reverse sweep and the partial sums for each of the 8
    # windows of 1024 tokens, Phase 1 adjoint segments and their verify kernel
    # (21 a step); without a retention gate 19
    assert bench.backward_launches(w, {"r": 1}, sms=152) == 21
    assert bench.backward_launches(w, {"r": None}, sms=152) == 19


FAKE = 0x10000  # never dereferenced: every case below fails validation first


def scan(L, io=1, B=1, H=1, T=8, K=64, k=FAKE, beta=FAKE, r=None, d0=None, kt=2 * FAKE,
         dT=None, ws=3 * FAKE, wsb=256):
    return L.osdn_precond_scan(io, B, H, T, K, k, beta, r, 0.1, d0, kt, dT, ws, wsb, None)


def chunk(L, io=1, B=1, H=1, T=8, K=64, V=64, q=FAKE, k=2 * FAKE, kt=3 * FAKE, v=4 * FAKE,
          beta=5 * FAKE, alpha=None, S0=None, o=6 * FAKE, ST=None, ws=7 * FAKE, wsb=None):
    if wsb is None:   # exactly what the shape needs
        wsb = L.osdn_chunk_fwd_workspace_bytes(io, B, H, T, K, V)
    return L.osdn_chunk_fwd(io, B, H, T, K, V, q, k, kt, v, beta, alpha, S0, o, ST, ws, wsb, None)


def test_host_validation_precond_scan(L):
    assert scan(L, io=7) == -3
    assert scan(L, K=96) == -2 and scan(L, K=32) == -2 and scan(L, T=-1) == -2
    assert scan(L, ws=None) == -5 and scan(L, wsb=8) == -5
    assert scan(L, k=None) == -1 and scan(L, beta=None) == -1 and scan(L, kt=None) == -1
    assert scan(L, k=FAKE + 4) == -4 and scan(L, d0=FAKE + 8) == -4
    assert scan(L, kt=FAKE) == -9          # ktilde aliases k
    assert scan(L, ws=FAKE) == -9          # the workspace overlaps k
    assert scan(L, ws=2 * FAKE - 128) == -9   # ... runs into ktilde
    assert scan(L, B=0) == 0               # empty batch: nothing to do


def resid(L, io=1, B=1, H=1, T=8, K=64, k=FAKE, kt=2 * FAKE, lr=4 * FAKE, ws=3 * FAKE, wsb=256):
    return L.osdn_precond_scan_residual(io, B, H, T, K, k, FAKE, None, 0.1, None, kt, None, lr,
                                        ws, wsb, None)


def test_host_validation_precond_scan_residual(L):
    assert resid(L, lr=None) == -1           # the diagnostic output is this call's point
    assert resid(L, io=7) == -3 and resid(L, K=96) == -2
    assert resid(L, lr=4 * FAKE + 4) == -4
    assert resid(L, lr=FAKE) == -9           # log_ratio overlaps k
    assert resid(L, lr=2 * FAKE) == -9       # log_ratio overlaps ktilde
    assert resid(L, B=0) == 0


def test_host_validation_chunk_fwd(L):
    assert chunk(L, io=2) == -3
    assert chunk(L, V=32) == -2 and chunk(L, H=-2) == -2
    assert chunk(L, q=None) == -1 and chunk(L, o=None) == -1
    assert chunk(L, v=4 * FAKE + 2) == -4
    assert chunk(L, o=FAKE) == -9          # o aliases q
    assert chunk(L, ws=6 * FAKE) == -9     # the workspace overlaps o
    assert chunk(L, ws=FAKE) == -9         # ... or an input
    assert chunk(L, wsb=0) == -5
    need = L.osdn_chunk_fwd_workspace_bytes(1, 1, 1, 8, 64, 64)
    assert chunk(L, wsb=need - 1) == -5
    assert chunk(L, H=0) == 0
    assert chunk(L, B=4096, H=4097) == -2  # more than 2^24 sequences
    # the tensor-core path's 32-bit chunk-row coordinates cap T; fp32 I/O has no cap
    cap = (0x7fffffff // 128) * 64
    assert chunk(L, T=cap + 1, wsb=1 << 62) == -2
    assert chunk(L, T=0x7fffffff, wsb=1 << 62) == -2
    assert chunk(L, io=0, T=cap + 1, wsb=1 << 62) != -2
    assert L.osdn_chunk_fwd_workspace_bytes(1, 1, 1, cap + 1, 128, 128) == 256
    assert L.osdn_chunk_fwd_workspace_bytes(1, 1, 1, cap, 128, 128) > 1 << 40


def test_chunk_fwd_workspace_size(L):
    # fp32 I/O and empty sequences need only the status word; bf16 keeps each
    # chunk's prepared operands: W (K x 64) and M (K x K) per chunk, Qe (2K
    # bytes a row) and Ae (128 bytes a row) on the chunk-padded length, g_C
    # per chunk, two fp32 states carried between slabs of chunks, and, where
    # the chain can run in time segments (as many as keep one chain CTA per
    # SM of 152, at least 16 chunks each), each segment's start and end state
    assert L.osdn_chunk_fwd_workspace_bytes(0, 2, 3, 100, 128, 64) == 256
    assert L.osdn_chunk_fwd_workspace_bytes(1, 2, 3, 0, 128, 64) == 256
    for B, H, T, K, V in [(1, 1, 1, 64, 64), (2, 3, 100, 128, 64), (1, 16, 65536, 128, 64),
                          (1, 16, 65536, 128, 128), (64, 32, 8192, 128, 128), (1, 2, 3217, 64, 64)]:
        BH, Tp, nch = B * H, -(-T // 64) * 64, -(-T // 64)
        r = lambda x: -(-x // 256) * 256
        nseg = max(1, min(152 // (BH * V // 64), nch // 16))
        seg = 2 * r(nseg * BH * V * K * 4) if nseg > 1 else 0
        want = (256 + r(BH * nch * K * 64 * 2) + r(BH * nch * K * K * 2) + r(BH * Tp * K * 2)
                + r(BH * Tp * 64 * 2) + r(BH * nch * 4) + 2 * r(BH * V * K * 4) + seg)
        assert L.osdn_chunk_fwd_workspace_bytes(1, B, H, T, K, V) == want, (B, H, T, K, V)


def fwd(L, io=1, B=1, H=1, T=8, K=64, V=64, q=FAKE, k=2 * FAKE, v=3 * FAKE, beta=4 * FAKE,
        r=None, d0=None, alpha=None, S0=None, o=5 * FAKE, dT=None, ST=None, ws=6 * FAKE, wsb=None):
    if wsb is None:   # exactly what the shape needs
        wsb = L.osdn_forward_workspace_bytes(io, B, H, T, K, V)
    return L.osdn_forward(io, B, H, T, K, V, q, k, v, beta, r, 0.1, d0, alpha, S0, o, dT, ST, ws,
                          wsb, None)


def test_host_validation_forward(L):
    assert fwd(L, io=2) == -3
    assert fwd(L, K=96) == -2 and fwd(L, V=32) == -2 and fwd(L, T=-1) == -2
    assert fwd(L, B=4096, H=4097) == -2      # more than 2^24 sequences
    assert fwd(L, ws=None) == -5 and fwd(L, wsb=8) == -5
    need = L.osdn_forward_workspace_bytes(1, 1, 1, 8, 64, 64)
    assert fwd(L, wsb=need - 1) == -5
    assert fwd(L, q=None) == -1 and fwd(L, k=None) == -1 and fwd(L, v=None) == -1
    assert fwd(L, beta=None) == -1 and fwd(L, o=None) == -1
    assert fwd(L, v=3 * FAKE + 2) == -4 and fwd(L, dT=7 * FAKE + 4) == -4
    assert fwd(L, o=FAKE) == -9              # o aliases q
    assert fwd(L, dT=2 * FAKE) == -9         # d_T aliases k
    assert fwd(L, ST=5 * FAKE) == -9         # S_T aliases o
    assert fwd(L, ws=FAKE) == -9             # the workspace overlaps q
    assert fwd(L, ws=5 * FAKE - 64) == -9    # ... runs into o
    assert fwd(L, H=0) == 0                  # empty batch: nothing to do
    cap = (0x7fffffff // 128) * 64           # the tensor-core Phase 2's cap on T
    assert fwd(L, T=cap + 1, wsb=1 << 62) == -2
    assert fwd(L, io=0, T=cap + 1, wsb=1 << 62) != -2


def test_forward_workspace_size(L):
    # bf16: the scan's segment scratch, e_t (4 bytes a token), d at every 64th
    # token (4 K bytes), then osdn_chunk_fwd's workspace; fp32: the scan's
    # scratch and ktilde in fp32; each part rounded up to 256 bytes
    r = lambda x: -(-x // 256) * 256
    assert L.osdn_forward_workspace_bytes(1, 2, 3, 0, 128, 64) == 256
    for B, H, T, K, V in [(1, 1, 1, 64, 64), (2, 3, 100, 128, 64), (2, 16, 8192, 128, 128),
                          (1, 16, 65536, 128, 128), (1, 2, 3217, 64, 64)]:
        BH = B * H
        p1 = L.osdn_precond_scan_workspace_bytes(B, H, T, K) - 256
        p2 = L.osdn_chunk_fwd_workspace_bytes(1, B, H, T, K, V) - 256
        want = 256 + r(p1) + r(BH * T * 4) + r(BH * (-(-T // 64)) * K * 4) + r(p2)
        assert L.osdn_forward_workspace_bytes(1, B, H, T, K, V) == want, (B, H, T, K, V)
        assert L.osdn_forward_workspace_bytes(0, B, H, T, K, V) == 256 + r(p1) + r(BH * T * K * 4)


def test_no_gpu_means_cuda_error_not_crash(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert scan(L) in (-6, -10)
    assert chunk(L) in (-6, -10)
    assert fwd(L) in (-6, -10)


def decode(L, io=1, B=1, H=1, K=64, V=64, q=FAKE, k=2 * FAKE, v=3 * FAKE, beta=4 * FAKE, r=None,
           alpha=None, d=5 * FAKE, S=6 * FAKE, o=7 * FAKE, kt=None, ws=8 * FAKE, wsb=256):
    return L.osdn_decode_step(io, B, H, K, V, q, k, v, beta, r, 0.1, alpha, d, S, o, kt, ws, wsb,
                              None)


def test_host_validation_decode_step(L):
    assert decode(L, io=3) == -3
    assert decode(L, K=32) == -2 and decode(L, V=96) == -2 and decode(L, B=-1) == -2
    assert decode(L, q=None) == -1 and decode(L, d=None) == -1 and decode(L, S=None) == -1
    assert decode(L, ws=None) == -5 and decode(L, wsb=16) == -5
    assert decode(L, k=2 * FAKE + 4) == -4
    assert decode(L, o=FAKE) == -9          # o aliases q
    assert decode(L, S=5 * FAKE) == -9      # S overlaps d
    assert decode(L, ws=7 * FAKE) == -9     # the workspace overlaps o
    assert decode(L, ws=2 * FAKE) == -9     # ... or an input
    assert decode(L, H=0) == 0


def bwd(L, io=1, B=1, H=1, T=8, K=64, V=64, ins=None, outs=None, ws=40 * FAKE, wsb=None):
    # inputs q, k, ktilde, v, beta, r, d0, alpha, S0, d_o, d_ST, d_dT, d_ktilde and
    # outputs dq, dk, dv, dbeta, dr, dalpha, dd0, dS0, deta at disjoint fake addresses
    a = {n: (i + 1) * FAKE for i, n in enumerate(
        ["q", "k", "kt", "v", "beta", "r", "d0", "alpha", "S0", "do", "dST", "ddT", "dkt",
         "dq", "dk", "dv", "dbeta", "dr", "dalpha", "dd0", "dS0", "deta"])}
    a.update(ins or {})
    a.update(outs or {})
    if wsb is None:
        wsb = L.osdn_backward_workspace_bytes(B, H, T, K, V)
    return L.osdn_backward(io, B, H, T, K, V, a["q"], a["k"], a["kt"], a["v"], a["beta"], a["r"],
                           0.1, a["d0"], a["alpha"], a["S0"], a["do"], a["dST"], a["ddT"],
                           a["dkt"], a["dq"], a["dk"], a["dv"], a["dbeta"], a["dr"], a["dalpha"],
                           a["dd0"], a["dS0"], a["deta"], ws, wsb, None)


def test_host_validation_backward(L):
    assert bwd(L, io=5) == -3
    assert bwd(L, K=96) == -2 and bwd(L, V=32) == -2 and bwd(L, T=-3) == -2
    assert bwd(L, B=4096, H=4097) == -2
    assert bwd(L, ws=None) == -5 and bwd(L, wsb=16) == -5
    need = L.osdn_backward_workspace_bytes(1, 1, 8, 64, 64)
    assert bwd(L, wsb=need - 1) == -5
    for n in ("q", "k", "kt", "v", "beta"):
        assert bwd(L, ins={n: None}) == -1, n
    for n in ("dq", "dk", "dv", "dbeta"):
        assert bwd(L, outs={n: None}) == -1, n
    assert bwd(L, ins={"alpha": 8 * FAKE + 4}) == -4
    assert bwd(L, outs={"deta": 22 * FAKE + 8}) == -4
    assert bwd(L, outs={"dq": FAKE}) == -9              # dq aliases q
    assert bwd(L, outs={"dS0": 11 * FAKE}) == -9        # dS0 aliases the cotangent d_ST
    assert bwd(L, outs={"dr": 17 * FAKE + 16}) == -9    # dr overlaps dbeta (8 tokens, 32 bytes)
    assert bwd(L, outs={"dr": 17 * FAKE + 32}) != -9    # ... and starts right after it
    assert bwd(L, ws=14 * FAKE) == -9                   # the workspace overlaps dq
    assert bwd(L, ws=FAKE) == -9                        # ... or an input
    assert bwd(L, ws=22 * FAKE - 64) == -9              # ... runs into deta
    assert bwd(L, H=0) == 0


def test_backward_workspace_size(L):
    # the state of each value row every 16 tokens, one partial of the row sums
    # (3K + 2 values a token) per block of 8 rows for one window of up to 1024
    # tokens, the state gradient carried between windows, Phase 1's inputs and
    # checkpoints, the forward scan's segment scratch (as osdn_precond_scan's),
    # and per time segment of the adjoint two K-vectors and two words; each
    # array padded to 256 bytes
    import bench
    r = lambda x: -(-x // 256) * 256
    assert L.osdn_backward_workspace_bytes(1, 2, 0, 64, 64) == 256
    for B, H, T, K, V in [(1, 1, 1, 64, 64), (2, 3, 100, 128, 64), (2, 16, 8192, 128, 128),
                          (1, 4, 3000, 64, 64)]:
        BH, ns = B * H, -(-T // 16)
        n = BH * bench.precond_segments(BH, T, True, 152)
        p1 = L.osdn_precond_scan_workspace_bytes(B, H, T, K) - 256
        tw = min(T, 1024)
        want = (256 + r(BH * ns * V * K * 4) + r(BH * (V // 8) * tw * (3 * K + 2) * 4)
                + r(BH * V * K * 4) + 2 * r(BH * T * K * 4) + r(BH * T * 4)
                + r(BH * ns * K * 4) + r(p1) + 2 * r(n * K * 4) + 2 * r(n * 4))
        assert L.osdn_backward_workspace_bytes(B, H, T, K, V) == want, (B, H, T, K, V)


def kda(L, io=1, B=1, H=1, T=8, K=64, V=64, q=FAKE, k=2 * FAKE, kt=3 * FAKE, v=4 * FAKE,
        beta=5 * FAKE, ak=None, S0=None, o=6 * FAKE, ST=None, ws=64 * FAKE, wsb=None):
    if wsb is None:   # exactly what the shape needs (more than FAKE bytes for bf16)
        wsb = L.osdn_chunk_fwd_kda_workspace_bytes(io, B, H, T, K, V)
    return L.osdn_chunk_fwd_kda(io, B, H, T, K, V, q, k, kt, v, beta, ak, S0, o, ST, ws, wsb,
                                None)


def test_chunk_fwd_kda_workspace_size(L):
    # fp32 I/O (the FFMA recurrence) needs only the status word; bf16 needs
    # osdn_chunk_fwd's workspace with the chunk's decay product per channel
    # (K floats a chunk instead of one)
    r = lambda x: -(-x // 256) * 256
    assert L.osdn_chunk_fwd_kda_workspace_bytes(0, 2, 16, 8192, 128, 128) == 256
    assert L.osdn_chunk_fwd_kda_workspace_bytes(1, 2, 16, 0, 128, 128) == 256
    for B, H, T, K, V in [(2, 16, 8192, 128, 128), (1, 2, 100, 64, 128), (1, 16, 65536, 128, 64)]:
        BH, nch = B * H, -(-T // 64)
        want = (L.osdn_chunk_fwd_workspace_bytes(1, B, H, T, K, V) - r(BH * nch * 4)
                + r(BH * nch * K * 4))
        assert L.osdn_chunk_fwd_kda_workspace_bytes(1, B, H, T, K, V) == want, (B, H, T, K, V)


def test_host_validation_chunk_fwd_kda(L):
    assert kda(L, io=2) == -3
    assert kda(L, K=32) == -2 and kda(L, V=96) == -2 and kda(L, T=-1) == -2
    assert kda(L, ws=None) == -5 and kda(L, wsb=255) == -5
    need = L.osdn_chunk_fwd_kda_workspace_bytes(1, 1, 1, 8, 64, 64)
    assert need > 256 and kda(L, wsb=need - 1) == -5
    cap = (0x7fffffff // 128) * 64           # the tensor-core path's cap on T
    assert kda(L, T=cap + 1, wsb=1 << 62) == -2
    assert kda(L, io=0, T=cap + 1, wsb=1 << 62) != -2
    assert kda(L, q=None) == -1 and kda(L, o=None) == -1 and kda(L, beta=None) == -1
    assert kda(L, ak=8 * FAKE + 4) == -4
    assert kda(L, o=FAKE) == -9                   # o aliases q
    assert kda(L, ws=6 * FAKE) == -9              # the workspace overlaps o
    assert kda(L, ws=4 * FAKE) == -9              # ... or an input
    # alpha_k is [B][H][T][K] fp32: 8 tokens x 64 channels = 2048 bytes
    assert kda(L, ak=8 * FAKE, o=8 * FAKE + 2032) == -9
    assert kda(L, ak=8 * FAKE, o=8 * FAKE + 2048) != -9
    assert kda(L, H=0) == 0


def test_host_validation_backward_kda(L):
    def call(**kw):
        ak = kw.pop("ak", 8 * FAKE)
        dak = kw.pop("dak", 19 * FAKE)
        a = {n: (i + 1) * FAKE for i, n in enumerate(
            ["q", "k", "kt", "v", "beta", "r", "d0", "alpha", "S0", "do", "dST", "ddT", "dkt",
             "dq", "dk", "dv", "dbeta", "dr", "dalpha", "dd0", "dS0", "deta"])}
        T, K, V = 8, 64, 64
        wsb = kw.pop("wsb", L.osdn_backward_kda_workspace_bytes(1, 1, T, K, V))
        return L.osdn_backward_kda(kw.pop("io", 1), 1, 1, T, K, V, a["q"], a["k"], a["kt"],
                                   a["v"], a["beta"], a["r"], 0.1, a["d0"], ak, a["S0"], a["do"],
                                   a["dST"], a["ddT"], a["dkt"], a["dq"], a["dk"], a["dv"],
                                   a["dbeta"], a["dr"], dak, a["dd0"], a["dS0"], a["deta"],
                                   40 * FAKE, wsb, None)
    assert call(io=4) == -3
    assert call(wsb=L.osdn_backward_workspace_bytes(1, 1, 8, 64, 64)) == -5  # too small here
    # dalpha_k is [T][K] fp32 (2048 bytes): it overlaps the next 2 KB, not a [T] vector's 32 B
    assert call(dak=19 * FAKE, ak=19 * FAKE + 1024) == -9
    assert call(dak=20 * FAKE - 1024) == -9                 # runs into dd0 at 20 * FAKE
    assert call() != -9 and call() != -2


def test_backward_kda_workspace_size(L):
    # as osdn_backward's, with the row-block partials carrying 4K + 1 values
    import bench
    r = lambda x: -(-x // 256) * 256
    for B, H, T, K, V in [(1, 1, 1, 64, 64), (2, 3, 100, 128, 64), (1, 4, 3000, 64, 64)]:
        BH, ns = B * H, -(-T // 16)
        n = BH * bench.precond_segments(BH, T, True, 152)
        p1 = L.osdn_precond_scan_workspace_bytes(B, H, T, K) - 256
        tw = min(T, 1024)
        want = (256 + r(BH * ns * V * K * 4) + r(BH * (V // 8) * tw * (4 * K + 1) * 4)
                + r(BH * V * K * 4) + 2 * r(BH * T * K * 4) + r(BH * T * 4)
                + r(BH * ns * K * 4) + r(p1) + 2 * r(n * K * 4) + 2 * r(n * 4))
        assert L.osdn_backward_kda_workspace_bytes(B, H, T, K, V) == want


def test_host_validation_decode_step_kda(L):
    def dk(**kw):
        a = dict(io=1, B=1, H=1, K=64, V=64, q=FAKE, k=2 * FAKE, v=3 * FAKE, beta=4 * FAKE,
                 r=None, ak=9 * FAKE, d=5 * FAKE, S=6 * FAKE, o=7 * FAKE, kt=None, ws=8 * FAKE,
                 wsb=256)
        a.update(kw)
        return L.osdn_decode_step_kda(a["io"], a["B"], a["H"], a["K"], a["V"], a["q"], a["k"],
                                      a["v"], a["beta"], a["r"], 0.1, a["ak"], a["d"], a["S"],
                                      a["o"], a["kt"], a["ws"], a["wsb"], None)
    assert dk(io=3) == -3 and dk(K=96) == -2 and dk(ws=None) == -5
    assert dk(q=None) == -1 and dk(ak=9 * FAKE + 8) == -4
    # alpha_k is [B][H][K] fp32 (256 bytes here), not one value per sequence
    assert dk(d=9 * FAKE + 128) == -9
    assert dk(d=9 * FAKE + 256) != -9
    assert dk(B=0) == 0
