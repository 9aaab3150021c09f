"""Shared helpers for the tests: error metric, oracle and GPU runners."""
import numpy as np
import torch

import oracle
from preconditioned_delta_rule_phase1_gb300 import synth

# Tolerances of the normwise max relative error max|x - ref| / max|ref|:
# fp32 I/O runs in fp32 FFMA; bf16 I/O rounds the operands of the tensor-core
# products to bf16 (unit roundoff 2^-9) and accumulates in fp32.
TOL = {"f32": 1e-4, "bf16": 2e-2}


def rel_err(x, ref) -> float:
    x = x.detach().double().cpu().numpy() if isinstance(x, torch.Tensor) else np.asarray(x)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    denom = max(float(np.max(np.abs(ref))), 1e-30)
    return float(np.max(np.abs(x - ref))) / denom


def to_cuda(x: dict) -> dict:
    return {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}


def oracle_forward(x: dict, heads=None):
    """fp64 oracle on all sequences, or on the flat sequence indices `heads`."""
    if heads is not None:
        x = synth.slice_heads(x, heads)
    return oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["r"], x["eta"], x["d0"],
                          x["alpha"], x["S0"])


def pick(t: torch.Tensor, heads):
    """GPU tensor [B,H,...] restricted to flat sequence indices, as [1,n,...]."""
    flat = t.reshape(-1, *t.shape[2:])
    return flat[list(heads)].unsqueeze(0)
