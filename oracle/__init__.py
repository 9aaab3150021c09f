"""fp64 CPU oracle for the OSDN forward pass (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library
and its Python binding) never loads it, and it shares no code with them.

The arithmetic lives in ``osdn_oracle.c`` (plain C, fp64, token by token),
which cites the passages of "OSDN: Improving Delta Rule with Provable Online
Preconditioning in Linear Attention" (gist.science summary pages, sections
1, 2.1, 2.2 and 2.3) that each step follows.  This module only compiles it
and marshals numpy arrays in and out.

``oracle/backward.py`` adds reference gradients (fp64 autograd through a
token-by-token torch restatement of the same recurrence), pinned by
``tests/test_oracle_backward.py`` against finite differences of this module's
forward.

Every function is pinned by ``tests/test_oracle_pins.py`` against facts the
pages and the mathematics fix (DeltaNet special case, definitional
hypergradient surrogate, residual-ratio identity and its per-sequence log sum,
dense unrolled product,
gated Newton condition, one-hot closed form, eta = 0 decay, state chaining).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "osdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libosdn_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no -march flags: it runs on x86 and Arm)."""
    with _lock:
        fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
        if fresh and not force:
            return _LIB_PATH
        os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        path = build()
        lib = ctypes.CDLL(path)
        lib.oracle_precond_scan.restype = ctypes.c_int
        lib.oracle_precond_scan.argtypes = [ctypes.c_int] * 4 + [_dp, _dp, _dp, ctypes.c_double,
                                                                 _dp, _dp, _dp, _dp, ctypes.c_int]
        lib.oracle_delta_fwd.restype = ctypes.c_int
        lib.oracle_delta_fwd.argtypes = [ctypes.c_int] * 5 + [_dp] * 9 + [ctypes.c_int]
        lib.oracle_delta_fwd_kda.restype = ctypes.c_int
        lib.oracle_delta_fwd_kda.argtypes = [ctypes.c_int] * 5 + [_dp] * 9 + [ctypes.c_int]
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # a torch tensor: upcast its exact stored values
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def precond_scan(k, beta, r=None, eta=0.1, d0=None, nthreads=None, log_ratio=False):
    """Phase 1: ktilde [B,H,T,K] and d_T [B,H,K] from k [B,H,T,K], beta [B,H,T].

    r [B,H,T] (None: r = 1) and d0 [B,H,K] (None: d0 = 1) are optional.
    With log_ratio=True also returns [B,H]: sum_t log((1 - beta_t <d_t, k_t^2>)^2),
    the log of the product of the token residual ratios f_t(S_t)/f_t(S_{t-1})
    (theorem 5.2; exp of it over T is the geometric-mean ratio q_geo).
    """
    k = _f64(k)
    B, H, T, K = k.shape
    beta, r, d0 = _f64(beta), _f64(r), _f64(d0)
    assert beta.shape == (B, H, T)
    assert r is None or r.shape == (B, H, T)
    assert d0 is None or d0.shape == (B, H, K)
    kt = np.empty_like(k)
    dT = np.empty((B, H, K))
    lr = np.empty((B, H)) if log_ratio else None
    rc = _load().oracle_precond_scan(B, H, T, K, _ptr(k), _ptr(beta), _ptr(r), float(eta),
                                     _ptr(d0), _ptr(kt), _ptr(dT), _ptr(lr),
                                     int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_precond_scan failed (%d)" % rc)
    return (kt, dT, lr) if log_ratio else (kt, dT)


def delta_fwd(q, k, ktilde, v, beta, alpha=None, S0=None, nthreads=None):
    """Phase 2: o [B,H,T,V] and S_T [B,H,V,K] by the token recurrence.

    alpha [B,H,T] (None: no decay) and S0 [B,H,V,K] (None: zeros) are optional.
    """
    q, k, ktilde, v = _f64(q), _f64(k), _f64(ktilde), _f64(v)
    B, H, T, K = k.shape
    V = v.shape[-1]
    beta, alpha, S0 = _f64(beta), _f64(alpha), _f64(S0)
    assert q.shape == k.shape == ktilde.shape and v.shape == (B, H, T, V)
    assert beta.shape == (B, H, T)
    assert alpha is None or alpha.shape == (B, H, T)
    assert S0 is None or S0.shape == (B, H, V, K)
    o = np.empty((B, H, T, V))
    ST = np.empty((B, H, V, K))
    rc = _load().oracle_delta_fwd(B, H, T, K, V, _ptr(q), _ptr(k), _ptr(ktilde), _ptr(v),
                                  _ptr(beta), _ptr(alpha), _ptr(S0), _ptr(o), _ptr(ST),
                                  int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_delta_fwd failed (%d)" % rc)
    return o, ST


def delta_fwd_kda(q, k, ktilde, v, beta, alpha_k=None, S0=None, nthreads=None):
    """Phase 2 with a per-channel decay (the Kimi-Delta-Attention-style gate):
    S_t = S_{t-1} Diag(alpha_t) + beta_t (v_t - S_{t-1} Diag(alpha_t) k_t) ktilde_t^T.

    alpha_k [B,H,T,K] (None: no decay) and S0 [B,H,V,K] are optional.
    Returns o [B,H,T,V] and S_T [B,H,V,K].
    """
    q, k, ktilde, v = _f64(q), _f64(k), _f64(ktilde), _f64(v)
    B, H, T, K = k.shape
    V = v.shape[-1]
    beta, alpha_k, S0 = _f64(beta), _f64(alpha_k), _f64(S0)
    assert q.shape == k.shape == ktilde.shape and v.shape == (B, H, T, V)
    assert beta.shape == (B, H, T)
    assert alpha_k is None or alpha_k.shape == (B, H, T, K)
    assert S0 is None or S0.shape == (B, H, V, K)
    o = np.empty((B, H, T, V))
    ST = np.empty((B, H, V, K))
    rc = _load().oracle_delta_fwd_kda(B, H, T, K, V, _ptr(q), _ptr(k), _ptr(ktilde), _ptr(v),
                                      _ptr(beta), _ptr(alpha_k), _ptr(S0), _ptr(o), _ptr(ST),
                                      int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_delta_fwd_kda failed (%d)" % rc)
    return o, ST


def forward_kda(q, k, v, beta, r=None, eta=0.1, d0=None, alpha_k=None, S0=None, nthreads=None):
    """Both phases with the per-channel decay in Phase 2 (Phase 1 unchanged).

    Returns (ktilde, dT, o, ST).
    """
    kt, dT = precond_scan(k, beta, r, eta, d0, nthreads)
    o, ST = delta_fwd_kda(q, k, kt, v, beta, alpha_k, S0, nthreads)
    return kt, dT, o, ST


def forward(q, k, v, beta, r=None, eta=0.1, d0=None, alpha=None, S0=None, nthreads=None):
    """Both phases in fp64: Phase 2 consumes the exact fp64 ktilde of Phase 1.

    Returns (ktilde, dT, o, ST).
    """
    kt, dT = precond_scan(k, beta, r, eta, d0, nthreads)
    o, ST = delta_fwd(q, k, kt, v, beta, alpha, S0, nthreads)
    return kt, dT, o, ST
