"""Thin ctypes binding of ``libosdn.so`` (include/osdn.h).

Argument marshalling only: every step of the forward pass and of its
gradients runs in the CUDA kernels behind the C ABI.  PyTorch provides device memory and the stream.
There is no CPU path: if the library is not built, or the tensors are not
on a CUDA device, the calls raise.

The C ABI takes plain pointers, so it cannot see shapes, dtypes or devices;
the binding checks them (every tensor's shape, dtype and device against the
call's layout) before any pointer leaves Python, and runs the call with the
tensors' device current and, by default, on its current stream.  A tensor
of the wrong type would otherwise be read or written out of its bounds.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

OSDN_F32, OSDN_BF16 = 0, 1
STATUS_BYTES = 256
_lock = threading.Lock()
_lib = None

_SIGS = {
    "osdn_version": (ctypes.c_int, []),
    "osdn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "osdn_precond_scan_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 4),
    "osdn_chunk_fwd_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 6),
    "osdn_workspace_init": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "osdn_check_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "osdn_precond_scan": (ctypes.c_int, [ctypes.c_int] * 5 + [ctypes.c_void_p] * 3 +
                          [ctypes.c_float] + [ctypes.c_void_p] * 4 +
                          [ctypes.c_size_t, ctypes.c_void_p]),
    "osdn_precond_scan_residual": (ctypes.c_int, [ctypes.c_int] * 5 + [ctypes.c_void_p] * 3 +
                                   [ctypes.c_float] + [ctypes.c_void_p] * 5 +
                                   [ctypes.c_size_t, ctypes.c_void_p]),
    "osdn_chunk_fwd": (ctypes.c_int, [ctypes.c_int] * 6 + [ctypes.c_void_p] * 10 +
                       [ctypes.c_size_t, ctypes.c_void_p]),
    "osdn_precond_scan_noalloc": (ctypes.c_int, [ctypes.c_int] * 5 + [ctypes.c_void_p] * 3 +
                                  [ctypes.c_float] + [ctypes.c_void_p] * 4),
    "osdn_decode_step": (ctypes.c_int, [ctypes.c_int] * 5 + [ctypes.c_void_p] * 5 +
                         [ctypes.c_float] + [ctypes.c_void_p] * 6 +
                         [ctypes.c_size_t, ctypes.c_void_p]),
    "osdn_backward_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 5),
    "osdn_backward": (ctypes.c_int, [ctypes.c_int] * 6 + [ctypes.c_void_p] * 6 +
                      [ctypes.c_float] + [ctypes.c_void_p] * 17 +
                      [ctypes.c_size_t, ctypes.c_void_p]),
    "osdn_backward_kda_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 5),
    "osdn_backward_kda": (ctypes.c_int, [ctypes.c_int] * 6 + [ctypes.c_void_p] * 6 +
                          [ctypes.c_float] + [ctypes.c_void_p] * 17 +
                          [ctypes.c_size_t, ctypes.c_void_p]),
    "osdn_decode_step_kda": (ctypes.c_int, [ctypes.c_int] * 5 + [ctypes.c_void_p] * 5 +
                             [ctypes.c_float] + [ctypes.c_void_p] * 6 +
                             [ctypes.c_size_t, ctypes.c_void_p]),
    "osdn_chunk_fwd_kda_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 6),
    "osdn_forward_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 6),
    "osdn_forward": (ctypes.c_int, [ctypes.c_int] * 6 + [ctypes.c_void_p] * 5 + [ctypes.c_float] +
                     [ctypes.c_void_p] * 7 + [ctypes.c_size_t, ctypes.c_void_p]),
    "osdn_chunk_fwd_kda": (ctypes.c_int, [ctypes.c_int] * 6 + [ctypes.c_void_p] * 10 +
                           [ctypes.c_size_t, ctypes.c_void_p]),
}


class OsdnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s (%d)" % (where, status_string(code), code))


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError("libosdn.so is not built (%s): run "
                                   "`python -m preconditioned_delta_rule_phase1_gb300.build`" % path)
            L = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype, fn.argtypes = res, args
            _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().osdn_status_string(int(code)).decode()


def _io(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return OSDN_F32
    if t.dtype == torch.bfloat16:
        return OSDN_BF16
    raise TypeError("io tensors must be float32 or bfloat16, got %s" % t.dtype)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("OSDN operates on CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("OSDN needs contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, device=None):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


F32 = torch.float32


def _expect(name, t, shape, dtype, device):
    """Raise unless `t` (a tensor, or None for an absent optional argument)
    has the shape, dtype and device the call reads or writes, and is dense."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor, got %s" % (name, type(t).__name__))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if t.dtype != dtype:
        raise TypeError("%s has dtype %s, expected %s" % (name, t.dtype, dtype))
    if t.device != device:
        raise ValueError("%s is on %s; the call runs on %s" % (name, t.device, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous (the library reads it densely)" % name)


def _on(device):
    """The context of a call on `device`: that CUDA device current."""
    if device.type != "cuda":
        raise ValueError("OSDN operates on CUDA tensors only")
    return torch.cuda.device(device)


def _workspace(workspace, device):
    ws = workspace or Workspace(device=device)
    if ws.buf.device != device:
        raise ValueError("workspace is on %s; the call runs on %s" % (ws.buf.device, device))
    return ws


def _check(code: int, where: str):
    if code != 0:
        raise OsdnError(code, where)


class Workspace:
    """A caller-owned device workspace (status word + per-call scratch)."""

    def __init__(self, nbytes: int = STATUS_BYTES, device=None, stream=None):
        self.device = torch.device(device or "cuda")
        self.buf = torch.empty(0, dtype=torch.uint8, device=self.device)
        self.ensure(max(nbytes, STATUS_BYTES), stream)

    def ensure(self, nbytes: int, stream=None):
        if self.buf.numel() < nbytes:
            old = self.buf
            self.buf = torch.zeros(((nbytes + 255) // 256) * 256, dtype=torch.uint8,
                                   device=self.device)
            if old.numel() >= STATUS_BYTES:  # keep a sticky status already raised
                self.buf[:STATUS_BYTES].copy_(old[:STATUS_BYTES])
        return self

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())

    @property
    def nbytes(self) -> int:
        return self.buf.numel()

    def reset(self, stream=None):
        _check(lib().osdn_workspace_init(self.ptr, self.nbytes, _stream(stream)), "workspace_init")

    def status(self, stream=None) -> int:
        return lib().osdn_check_status(self.ptr, _stream(stream))


def precond_scan_workspace_bytes(B, H, T, K) -> int:
    return int(lib().osdn_precond_scan_workspace_bytes(B, H, T, K))


def chunk_fwd_workspace_bytes(io, B, H, T, K, V) -> int:
    return int(lib().osdn_chunk_fwd_workspace_bytes(io, B, H, T, K, V))


def forward_workspace_bytes(io, B, H, T, K, V) -> int:
    return int(lib().osdn_forward_workspace_bytes(io, B, H, T, K, V))


def backward_workspace_bytes(B, H, T, K, V) -> int:
    return int(lib().osdn_backward_workspace_bytes(B, H, T, K, V))


def backward_kda_workspace_bytes(B, H, T, K, V) -> int:
    return int(lib().osdn_backward_kda_workspace_bytes(B, H, T, K, V))


def precond_scan(k, beta, r=None, eta=0.1, d0=None, ktilde=None, dT=None, workspace=None,
                 stream=None, log_ratio=None):
    """Phase 1 (osdn_precond_scan): returns (ktilde, dT).

    With ``log_ratio`` (True, or a [B, H] fp32 tensor to fill) the call goes
    through osdn_precond_scan_residual and returns (ktilde, dT, log_ratio):
    per sequence sum_t log((1 - beta_t <d_t, k_t^2>)^2).
    """
    B, H, T, K = k.shape
    io, dev = _io(k), k.device
    _expect("beta", beta, (B, H, T), F32, dev)
    _expect("r", r, (B, H, T), F32, dev)
    _expect("d0", d0, (B, H, K), F32, dev)
    if ktilde is None:
        ktilde = torch.empty_like(k)
    if dT is None:
        dT = torch.empty(B, H, K, dtype=F32, device=dev)
    _expect("ktilde", ktilde, (B, H, T, K), k.dtype, dev)
    _expect("dT", dT, (B, H, K), F32, dev)
    residual = not (log_ratio is None or log_ratio is False)
    if log_ratio is True:
        log_ratio = torch.empty(B, H, dtype=F32, device=dev)
    if residual:
        _expect("log_ratio", log_ratio, (B, H), F32, dev)
    ws = _workspace(workspace, dev)
    with _on(dev):
        ws.ensure(precond_scan_workspace_bytes(B, H, T, K))
        if not residual:
            code = lib().osdn_precond_scan(io, B, H, T, K, _ptr(k), _ptr(beta), _ptr(r),
                                           float(eta), _ptr(d0), _ptr(ktilde), _ptr(dT), ws.ptr,
                                           ws.nbytes, _stream(stream, dev))
            _check(code, "osdn_precond_scan")
            return ktilde, dT
        code = lib().osdn_precond_scan_residual(io, B, H, T, K, _ptr(k), _ptr(beta), _ptr(r),
                                                float(eta), _ptr(d0), _ptr(ktilde), _ptr(dT),
                                                _ptr(log_ratio), ws.ptr, ws.nbytes,
                                                _stream(stream, dev))
    _check(code, "osdn_precond_scan_residual")
    return ktilde, dT, log_ratio


def precond_scan_noalloc(k, beta, r=None, eta=0.1, d0=None, ktilde=None, dT=None, stream=None):
    """Phase 1 through osdn_precond_scan_noalloc: no workspace, no device
    allocation inside the call (outputs are allocated here only when not given)."""
    B, H, T, K = k.shape
    io, dev = _io(k), k.device
    _expect("beta", beta, (B, H, T), F32, dev)
    _expect("r", r, (B, H, T), F32, dev)
    _expect("d0", d0, (B, H, K), F32, dev)
    if ktilde is None:
        ktilde = torch.empty_like(k)
    if dT is None:
        dT = torch.empty(B, H, K, dtype=F32, device=dev)
    _expect("ktilde", ktilde, (B, H, T, K), k.dtype, dev)
    _expect("dT", dT, (B, H, K), F32, dev)
    with _on(dev):
        code = lib().osdn_precond_scan_noalloc(io, B, H, T, K, _ptr(k), _ptr(beta), _ptr(r),
                                               float(eta), _ptr(d0), _ptr(ktilde), _ptr(dT),
                                               _stream(stream, dev))
    _check(code, "osdn_precond_scan_noalloc")
    return ktilde, dT


def chunk_fwd(q, k, ktilde, v, beta, alpha=None, S0=None, o=None, ST=None, workspace=None,
              stream=None):
    """Phase 2 (osdn_chunk_fwd): returns (o, ST)."""
    B, H, T, K = k.shape
    V = v.shape[-1]
    io, dev = _io(k), k.device
    _expect("q", q, (B, H, T, K), k.dtype, dev)
    _expect("ktilde", ktilde, (B, H, T, K), k.dtype, dev)
    _expect("v", v, (B, H, T, V), k.dtype, dev)
    _expect("beta", beta, (B, H, T), F32, dev)
    _expect("alpha", alpha, (B, H, T), F32, dev)
    _expect("S0", S0, (B, H, V, K), F32, dev)
    if o is None:
        o = torch.empty(B, H, T, V, dtype=k.dtype, device=dev)
    if ST is None:
        ST = torch.empty(B, H, V, K, dtype=F32, device=dev)
    _expect("o", o, (B, H, T, V), k.dtype, dev)
    _expect("ST", ST, (B, H, V, K), F32, dev)
    ws = _workspace(workspace, dev)
    with _on(dev):
        ws.ensure(chunk_fwd_workspace_bytes(io, B, H, T, K, V))
        code = lib().osdn_chunk_fwd(io, B, H, T, K, V, _ptr(q), _ptr(k), _ptr(ktilde), _ptr(v),
                                    _ptr(beta), _ptr(alpha), _ptr(S0), _ptr(o), _ptr(ST), ws.ptr,
                                    ws.nbytes, _stream(stream, dev))
    _check(code, "osdn_chunk_fwd")
    return o, ST


def forward(q, k, v, beta, r=None, eta=0.1, d0=None, alpha=None, S0=None, workspace=None,
            stream=None):
    """Both phases: returns (ktilde, dT, o, ST)."""
    ws = _workspace(workspace, k.device)
    ktilde, dT = precond_scan(k, beta, r, eta, d0, workspace=ws, stream=stream)
    o, ST = chunk_fwd(q, k, ktilde, v, beta, alpha, S0, workspace=ws, stream=stream)
    return ktilde, dT, o, ST


def forward_fused(q, k, v, beta, r=None, eta=0.1, d0=None, alpha=None, S0=None, o=None, dT=None,
                  ST=None, workspace=None, stream=None):
    """Both phases in one call (osdn_forward), ktilde kept off global memory
    for bf16 I/O: returns (dT, o, ST)."""
    B, H, T, K = k.shape
    V = v.shape[-1]
    io, dev = _io(k), k.device
    _expect("q", q, (B, H, T, K), k.dtype, dev)
    _expect("v", v, (B, H, T, V), k.dtype, dev)
    _expect("beta", beta, (B, H, T), F32, dev)
    _expect("r", r, (B, H, T), F32, dev)
    _expect("d0", d0, (B, H, K), F32, dev)
    _expect("alpha", alpha, (B, H, T), F32, dev)
    _expect("S0", S0, (B, H, V, K), F32, dev)
    if o is None:
        o = torch.empty(B, H, T, V, dtype=k.dtype, device=dev)
    if dT is None:
        dT = torch.empty(B, H, K, dtype=F32, device=dev)
    if ST is None:
        ST = torch.empty(B, H, V, K, dtype=F32, device=dev)
    _expect("o", o, (B, H, T, V), k.dtype, dev)
    _expect("dT", dT, (B, H, K), F32, dev)
    _expect("ST", ST, (B, H, V, K), F32, dev)
    ws = _workspace(workspace, dev)
    with _on(dev):
        ws.ensure(forward_workspace_bytes(io, B, H, T, K, V))
        code = lib().osdn_forward(io, B, H, T, K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(r),
                                  float(eta), _ptr(d0), _ptr(alpha), _ptr(S0), _ptr(o), _ptr(dT),
                                  _ptr(ST), ws.ptr, ws.nbytes, _stream(stream, dev))
    _check(code, "osdn_forward")
    return dT, o, ST


def decode_step(q, k, v, beta, d, S, r=None, eta=0.1, alpha=None, o=None, ktilde=None,
                workspace=None, stream=None):
    """One recurrent step (osdn_decode_step): updates d [B,H,K] and S [B,H,V,K]
    (fp32) in place for the token q, k [B,H,K], v [B,H,V] (io); returns
    (o, ktilde)."""
    return _decode(False, q, k, v, beta, d, S, r, eta, alpha, o, ktilde, workspace, stream)


def decode_step_kda(q, k, v, beta, d, S, r=None, eta=0.1, alpha_k=None, o=None, ktilde=None,
                    workspace=None, stream=None):
    """One recurrent step with a decay per key channel (osdn_decode_step_kda):
    as ``decode_step``, with alpha_k [B,H,K] fp32."""
    return _decode(True, q, k, v, beta, d, S, r, eta, alpha_k, o, ktilde, workspace, stream)


def _decode(per_channel, q, k, v, beta, d, S, r, eta, alpha, o, ktilde, workspace, stream):
    B, H, K = k.shape
    V = v.shape[-1]
    io, dev = _io(k), k.device
    _expect("q", q, (B, H, K), k.dtype, dev)
    _expect("v", v, (B, H, V), k.dtype, dev)
    _expect("beta", beta, (B, H), F32, dev)
    _expect("r", r, (B, H), F32, dev)
    _expect("alpha", alpha, (B, H, K) if per_channel else (B, H), F32, dev)
    _expect("d", d, (B, H, K), F32, dev)
    _expect("S", S, (B, H, V, K), F32, dev)
    if o is None:
        o = torch.empty(B, H, V, dtype=k.dtype, device=dev)
    if ktilde is None:
        ktilde = torch.empty(B, H, K, dtype=k.dtype, device=dev)
    _expect("o", o, (B, H, V), k.dtype, dev)
    _expect("ktilde", ktilde, (B, H, K), k.dtype, dev)
    ws = _workspace(workspace, dev)
    name = "osdn_decode_step_kda" if per_channel else "osdn_decode_step"
    with _on(dev):
        code = getattr(lib(), name)(io, B, H, K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                    _ptr(r), float(eta), _ptr(alpha), _ptr(d), _ptr(S), _ptr(o),
                                    _ptr(ktilde), ws.ptr, ws.nbytes, _stream(stream, dev))
    _check(code, name)
    return o, ktilde


def backward(q, k, ktilde, v, beta, r=None, eta=0.1, d0=None, alpha=None, S0=None, *, do=None,
             dST=None, ddT=None, dktilde=None, workspace=None, stream=None):
    """Gradients of both phases (osdn_backward).

    Takes the forward's inputs, the ktilde it produced and the cotangents of
    its outputs (o, ST, dT, ktilde; None counts as zero).  Returns a dict
    keyed like the inputs: q, k, v, beta (io / fp32), eta ([B, H]: each
    sequence's share; the scalar gradient is the sum), and r, alpha, d0, S0
    for those given (an input given as None has no entry).
    """
    return _backward(False, q, k, ktilde, v, beta, r, eta, d0, alpha, S0, do, dST, ddT, dktilde,
                     workspace, stream)


def backward_kda(q, k, ktilde, v, beta, r=None, eta=0.1, d0=None, alpha_k=None, S0=None, *,
                 do=None, dST=None, ddT=None, dktilde=None, workspace=None, stream=None):
    """Gradients of both phases with a decay per key channel
    (osdn_backward_kda): as ``backward``, with alpha_k [B, H, T, K] and its
    gradient under the key "alpha" ([B, H, T, K])."""
    return _backward(True, q, k, ktilde, v, beta, r, eta, d0, alpha_k, S0, do, dST, ddT,
                     dktilde, workspace, stream)


def _backward(per_channel, q, k, ktilde, v, beta, r, eta, d0, alpha, S0, do, dST, ddT, dktilde,
              workspace, stream):
    B, H, T, K = k.shape
    V = v.shape[-1]
    io, dev = _io(k), k.device
    ashape = (B, H, T, K) if per_channel else (B, H, T)
    for name, t, shape, dt in (("q", q, (B, H, T, K), k.dtype),
                               ("ktilde", ktilde, (B, H, T, K), k.dtype),
                               ("v", v, (B, H, T, V), k.dtype),
                               ("beta", beta, (B, H, T), F32), ("r", r, (B, H, T), F32),
                               ("d0", d0, (B, H, K), F32), ("alpha", alpha, ashape, F32),
                               ("S0", S0, (B, H, V, K), F32), ("do", do, (B, H, T, V), k.dtype),
                               ("dST", dST, (B, H, V, K), F32), ("ddT", ddT, (B, H, K), F32),
                               ("dktilde", dktilde, (B, H, T, K), k.dtype)):
        _expect(name, t, shape, dt, dev)
    if q is None or ktilde is None or v is None or beta is None:
        raise ValueError("q, ktilde, v and beta are required")
    new = lambda *shape, dtype=F32: torch.empty(*shape, dtype=dtype, device=dev)
    g = {"q": new(B, H, T, K, dtype=k.dtype), "k": new(B, H, T, K, dtype=k.dtype),
         "v": new(B, H, T, V, dtype=k.dtype), "beta": new(B, H, T), "eta": new(B, H)}
    if r is not None:
        g["r"] = new(B, H, T)
    if alpha is not None:
        g["alpha"] = new(*ashape)
    if d0 is not None:
        g["d0"] = new(B, H, K)
    if S0 is not None:
        g["S0"] = new(B, H, V, K)
    ws = _workspace(workspace, dev)
    fn, size = ((lib().osdn_backward_kda, backward_kda_workspace_bytes) if per_channel
                else (lib().osdn_backward, backward_workspace_bytes))
    with _on(dev):
        ws.ensure(size(B, H, T, K, V))
        code = fn(io, B, H, T, K, V, _ptr(q), _ptr(k), _ptr(ktilde), _ptr(v), _ptr(beta), _ptr(r),
                  float(eta), _ptr(d0), _ptr(alpha), _ptr(S0), _ptr(do), _ptr(dST), _ptr(ddT),
                  _ptr(dktilde), _ptr(g["q"]), _ptr(g["k"]), _ptr(g["v"]), _ptr(g["beta"]),
                  _ptr(g.get("r")), _ptr(g.get("alpha")), _ptr(g.get("d0")), _ptr(g.get("S0")),
                  _ptr(g["eta"]), ws.ptr, ws.nbytes, _stream(stream, dev))
    _check(code, "osdn_backward_kda" if per_channel else "osdn_backward")
    return g


def chunk_fwd_kda(q, k, ktilde, v, beta, alpha_k=None, S0=None, o=None, ST=None, workspace=None,
                  stream=None):
    """Phase 2 with a decay per key channel (osdn_chunk_fwd_kda), alpha_k
    [B, H, T, K] fp32: returns (o, ST)."""
    B, H, T, K = k.shape
    V = v.shape[-1]
    io, dev = _io(k), k.device
    _expect("q", q, (B, H, T, K), k.dtype, dev)
    _expect("ktilde", ktilde, (B, H, T, K), k.dtype, dev)
    _expect("v", v, (B, H, T, V), k.dtype, dev)
    _expect("beta", beta, (B, H, T), F32, dev)
    _expect("alpha_k", alpha_k, (B, H, T, K), F32, dev)
    _expect("S0", S0, (B, H, V, K), F32, dev)
    if o is None:
        o = torch.empty(B, H, T, V, dtype=k.dtype, device=dev)
    if ST is None:
        ST = torch.empty(B, H, V, K, dtype=F32, device=dev)
    _expect("o", o, (B, H, T, V), k.dtype, dev)
    _expect("ST", ST, (B, H, V, K), F32, dev)
    ws = _workspace(workspace, dev)
    with _on(dev):
        ws.ensure(int(lib().osdn_chunk_fwd_kda_workspace_bytes(io, B, H, T, K, V)))
        code = lib().osdn_chunk_fwd_kda(io, B, H, T, K, V, _ptr(q), _ptr(k), _ptr(ktilde),
                                        _ptr(v), _ptr(beta), _ptr(alpha_k), _ptr(S0), _ptr(o),
                                        _ptr(ST), ws.ptr, ws.nbytes, _stream(stream, dev))
    _check(code, "osdn_chunk_fwd_kda")
    return o, ST


def forward_kda(q, k, v, beta, r=None, eta=0.1, d0=None, alpha_k=None, S0=None, workspace=None,
                stream=None):
    """Both phases with a decay per key channel in Phase 2: returns
    (ktilde, dT, o, ST)."""
    ws = _workspace(workspace, k.device)
    ktilde, dT = precond_scan(k, beta, r, eta, d0, workspace=ws, stream=stream)
    o, ST = chunk_fwd_kda(q, k, ktilde, v, beta, alpha_k, S0, workspace=ws, stream=stream)
    return ktilde, dT, o, ST
