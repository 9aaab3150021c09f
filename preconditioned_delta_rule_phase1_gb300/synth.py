"""Seeded synthetic inputs for the OSDN forward pass.

This module holds no arithmetic of the method: it only draws the inputs
(keys, queries, values, gates, initial states) that both the CUDA path and
the fp64 oracle consume, so that both see byte-identical data.

Recipe (the pages measure on trained 340M / 1.3B models and recall suites
that cannot be run here; these seeded draws stand in for their layer shapes):

* q, k ~ N(0, 1) per element in fp32, then L2-normalised per head vector;
  v ~ N(0, 1); all three cast to the I/O dtype afterwards.
* beta = sigmoid(N(0, 1)) per token-head; retention r = sigmoid(N(2, 1)) per
  token-head when the adaptive-forgetting gate is on; decay
  alpha = exp(-0.1 * softplus(N(0, 1))) per token-head for the gated variant;
  S0 ~ N(0, 0.01) (standard deviation 0.01) where a non-zero start state is
  used.  Gates and states stay fp32.
* The repeated-key recall stream: the second half of each sequence reuses
  the first half's keys in a per-(b,h) random order, each plus
  N(0, 0.05) noise and renormalised (a synthetic stand-in for the
  "keys recur" recall setting of the pages' section 4.1).
* A torch CPU generator seeded once draws, in this fixed order:
  q, k, v, beta logits, r logits, alpha logits, S0, permutation, noise.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    io: str            # "f32" or "bf16"
    B: int
    H: int
    T: int
    K: int
    V: int
    eta: float
    apf: bool = False          # retention gate r on
    gated: bool = False        # per-token decay alpha on
    s0: bool = False           # non-zero start state
    repeat_keys: bool = False  # second half reuses the first half's keys
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def tokens(self) -> int:
        return self.B * self.T

    @property
    def token_heads(self) -> int:
        return self.B * self.H * self.T


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", "f32", 1, 2, 256, 64, 64, 0.1,
                         note="tiny fp32 OSDN, r=1, d0=1, S0=0"),
    "lm340m_bf16": Workload("lm340m_bf16", "bf16", 8, 8, 2048, 128, 128, 0.1,
                            note="340M-class layer shape, r=1"),
    "recall_apf_bf16": Workload("recall_apf_bf16", "bf16", 4, 16, 4096, 64, 64, 0.2, apf=True,
                                repeat_keys=True, note="repeated-key recall stream with APF"),
    "lm1p3b_apf_bf16": Workload("lm1p3b_apf_bf16", "bf16", 2, 16, 8192, 128, 128, 0.1, apf=True,
                                note="1.3B-class layer shape with APF"),
    "long_gated_apf_bf16": Workload("long_gated_apf_bf16", "bf16", 1, 16, 65536, 128, 128, 0.1,
                                    apf=True, gated=True, s0=True,
                                    note="long-context gated variant with APF, S0 ~ N(0, 0.01)"),
}
WORKLOAD_ORDER = ["tiny_f32", "lm340m_bf16", "recall_apf_bf16", "lm1p3b_apf_bf16",
                  "long_gated_apf_bf16"]


def torch_dtype(io: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[io]


def _normalise(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def make_inputs(w: Workload, seed: int | None = None) -> dict:
    """All inputs of workload ``w`` as CPU tensors (io dtype for q/k/v)."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    B, H, T, K, V = w.B, w.H, w.T, w.K, w.V
    q = _normalise(torch.randn(B, H, T, K, generator=g))
    k = torch.randn(B, H, T, K, generator=g)
    v = torch.randn(B, H, T, V, generator=g)
    beta = torch.sigmoid(torch.randn(B, H, T, generator=g))
    r = torch.sigmoid(torch.randn(B, H, T, generator=g) + 2.0) if w.apf else None
    alpha = (torch.exp(-0.1 * torch.nn.functional.softplus(torch.randn(B, H, T, generator=g)))
             if w.gated else None)
    S0 = torch.randn(B, H, V, K, generator=g) * 0.01 if w.s0 else None
    if w.repeat_keys:
        half = T // 2
        perm = torch.stack([torch.randperm(half, generator=g) for _ in range(B * H)])
        perm = perm.view(B, H, half)
        noise = torch.randn(B, H, T - half, K, generator=g) * 0.05
        base = _normalise(k[:, :, :half])
        src = torch.gather(base, 2, perm[..., None].expand(B, H, half, K))
        tail = src[:, :, : T - half] + noise
        k = torch.cat([base, tail], dim=2)
    k = _normalise(k)
    dt = torch_dtype(w.io)
    return {
        "q": q.to(dt).contiguous(), "k": k.to(dt).contiguous(), "v": v.to(dt).contiguous(),
        "beta": beta.contiguous(),
        "r": None if r is None else r.contiguous(),
        "alpha": None if alpha is None else alpha.contiguous(),
        "S0": None if S0 is None else S0.contiguous(),
        "d0": None, "eta": w.eta,
    }


def make_random(B, H, T, K, V, io="f32", apf=False, gated=False, s0=False, d0=False,
                eta=0.1, seed=0, repeat_keys=False) -> dict:
    """Inputs of an arbitrary shape drawn by the same recipe (edge-case tests)."""
    w = Workload("custom", io, B, H, T, K, V, eta, apf=apf, gated=gated, s0=s0,
                 repeat_keys=repeat_keys, seed=seed)
    x = make_inputs(w)
    if d0:
        g = torch.Generator().manual_seed(seed + 7919)
        x["d0"] = (0.5 + torch.rand(B, H, K, generator=g)).contiguous()
    return x


def slice_heads(x: dict, heads) -> dict:
    """The inputs restricted to a list of flat (b*H + h) sequence indices, as [1, n, ...]."""
    out = {}
    for name, t in x.items():
        if isinstance(t, torch.Tensor):
            flat = t.reshape(-1, *t.shape[2:])
            out[name] = flat[list(heads)].unsqueeze(0).contiguous()
        else:
            out[name] = t
    return out
