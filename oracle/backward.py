"""fp64 reference gradients of the OSDN forward pass (test infrastructure only).

Only the tests may import this module; nothing in the product path loads it,
and it shares no code with the CUDA library.

It restates the forward pass of both phases token by token with float64
PyTorch CPU ops -- the recurrence of ``osdn_oracle.c`` with the same readings
of the pages ("OSDN: Improving Delta Rule with Provable Online
Preconditioning in Linear Attention", gist.science summary, sections 2.1,
2.2 and 2.3):

    ktilde_t = d_t (.) k_t
    d_{t+1}  = r_t d_t + eta beta_t (1 - beta_t <d_t, k_t^2>) k_t^2 / ||k_t||^2
               (no step for a zero key)
    S_t      = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) ktilde_t^T
               (or, with a decay per key channel, S_{t-1} Diag(alpha_t) in
               place of alpha_t S_{t-1})
    o_t      = S_t q_t

and differentiates it with ``torch.autograd``: the gradients of a training
step are, by definition, the derivative of this forward, so the reference is
that derivative taken exactly (to fp64 rounding) rather than any chunked or
reordered backward recurrence.

Pinned by ``tests/test_oracle_backward.py``: its forward equals the C
oracle's, and its gradients equal central finite differences of the C
oracle's forward for every input.
"""
from __future__ import annotations

import torch

_F = torch.float64


def _t(x, requires_grad=False):
    if x is None:
        return None
    t = torch.as_tensor(x, dtype=_F).clone()
    return t.requires_grad_(requires_grad)


def forward_torch(q, k, v, beta, r=None, eta=0.1, d0=None, alpha=None, S0=None, ktilde=None):
    """Both phases, token by token, in float64 torch ops (differentiable).

    Shapes as in ``oracle.forward``; alpha may also be [B, H, T, K], a decay
    per key channel (``oracle.forward_kda``): S_t = S_{t-1} Diag(alpha_t) +
    beta_t (v_t - S_{t-1} Diag(alpha_t) k_t) ktilde_t^T.  Returns (ktilde, dT,
    o, ST).

    ``ktilde`` [B, H, T, K], if given, is the value Phase 2 uses in place of
    d_t (.) k_t -- the forward's stored keys, e.g. rounded to the I/O type --
    while the derivative still flows through d_t (.) k_t (a straight-through
    value).  The backward kernels take the stored ktilde, so this is the
    exact derivative of what they differentiate.
    """
    B, H, T, K = k.shape
    V = v.shape[-1]
    d = d0 if d0 is not None else torch.ones(B, H, K, dtype=_F)
    S = S0 if S0 is not None else torch.zeros(B, H, V, K, dtype=_F)
    kts, outs = [], []
    for t in range(T):
        kt = k[:, :, t]
        w = kt * kt
        n = w.sum(-1)
        a = (d * w).sum(-1)
        bt = beta[:, :, t]
        ktil = d * kt                                       # preconditioner before the step
        if ktilde is not None:                              # stored value, same derivative
            ktil = ktil + (ktilde[:, :, t] - ktil).detach()
        safe_n = torch.where(n > 0, n, torch.ones_like(n))
        coef = torch.where(n > 0, eta * bt * (1.0 - bt * a) / safe_n, torch.zeros_like(n))
        rt = r[:, :, t] if r is not None else torch.ones_like(bt)
        d = rt[..., None] * d + coef[..., None] * w         # descent step on h_t
        if alpha is None:
            Sbar = S
        elif alpha.dim() == 4:                               # per key channel
            Sbar = S * alpha[:, :, t][..., None, :]
        else:
            Sbar = alpha[:, :, t][..., None, None] * S
        Sk = torch.einsum("bhvk,bhk->bhv", Sbar, kt)        # alpha_t S_{t-1} k_t
        u = bt[..., None] * (v[:, :, t] - Sk)
        S = Sbar + u[..., :, None] * ktil[..., None, :]
        outs.append(torch.einsum("bhvk,bhk->bhv", S, q[:, :, t]))   # read-out after the write
        kts.append(ktil)
    return torch.stack(kts, 2), d, torch.stack(outs, 2), S


def grads(q, k, v, beta, r=None, eta=0.1, d0=None, alpha=None, S0=None, *, do=None, ddT=None,
          dST=None, dkt=None, ktilde=None):
    """Gradients of L = <o, do> + <d_T, ddT> + <S_T, dST> + <ktilde, dkt> with
    respect to every input (the cotangents that are None count as zero);
    ``ktilde`` as in ``forward_torch`` (the stored keys Phase 2 uses).

    Returns a dict keyed like the inputs (q, k, v, beta, r, eta, d0, alpha,
    S0); an input given as None has no entry.  eta's entry is a float.
    """
    ins = {"q": _t(q, True), "k": _t(k, True), "v": _t(v, True), "beta": _t(beta, True),
           "r": _t(r, True), "eta": _t(eta, True), "d0": _t(d0, True), "alpha": _t(alpha, True),
           "S0": _t(S0, True)}
    kt, dT, o, ST = forward_torch(ins["q"], ins["k"], ins["v"], ins["beta"], ins["r"], ins["eta"],
                                  ins["d0"], ins["alpha"], ins["S0"], _t(ktilde))
    loss = torch.zeros((), dtype=_F)
    for out, cot in ((o, do), (dT, ddT), (ST, dST), (kt, dkt)):
        if cot is not None:
            loss = loss + (out * _t(cot)).sum()
    names = [n for n, x in ins.items() if x is not None]
    gs = torch.autograd.grad(loss, [ins[n] for n in names], allow_unused=True)
    res = {}
    for n, g in zip(names, gs):
        g = torch.zeros_like(ins[n]) if g is None else g
        res[n] = float(g) if n == "eta" else g.detach().numpy()
    return res
