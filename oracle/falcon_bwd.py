"""Gradients of the Falcon forward pass: fp64 autograd over the token-by-token recurrence.

TEST INFRASTRUCTURE. This is the reference the CUDA backward kernels are checked against. Only the
tests, the smoke check and the benchmark's CPU-baseline leg may import it; it shares no code with
the CUDA path.

The forward recurrence is written out with plain PyTorch CPU operations in fp64, one token at a
time, as the C oracle computes it ("Fast Weight Attention for Continual Learning": paperlayer
summary §3, §3.1, §C.3, §4.6, Appendix p.34; agihunt explainer "Method"):
    x_tau = k_{tau-1} (x_1 = 0; the tail key k_pos when the call continues at pos > 0), y_tau = v_tau
    eta = beta / (||x||^2 + lambda + eps)   (0 when the denominator is 0, and at tau = 1)
    alpha = min(eta lambda, 1 - eps_gamma)  (0 at tau = 1), gamma = 1 - alpha
    Falcon-1:  S = gamma S + eta x (y - S^T x)^T      Falcon-1A: S = gamma S + eta x y^T
    Falcon-2, 2A: the same per value column c, with beta[..., c] (so eta, alpha per column)
    o_tau = S_tau^T q_tau
and torch.autograd differentiates it. Two points of the pages' backward follow from this definition
and are written so that autograd takes them exactly (paperlayer §D.2, §E.3, §G.3):
  * the clamp: the adjoint of alpha passes only where eta lambda < 1 - eps_gamma (the unclamped
    indicator); where the clamp binds, alpha is the constant 1 - eps_gamma;
  * the zero step: where eta is 0 by definition (zero denominator, tau = 1) no gradient reaches
    beta, lambda or x through eta (no 0/0 is formed).
The first step of a fresh sequence (tau = 1) carries no gradient to its beta and lambda (the pages'
boundary constants). The gradient returned for `tail` is that of the pending key k_pos.
"""

from __future__ import annotations

import numpy as np
import torch

FALCON_1, FALCON_1A, FALCON_2, FALCON_2A = 1, 2, 3, 4


def forward_torch(variant, q, k, v, beta, lam, S0=None, *, pos=0, tail=None, eps=1e-6, eps_gamma=1e-6):
    """The recurrence on fp64 torch tensors (autograd-capable). q, k [B,H,T,dk], v [B,H,T,dv],
    beta [B,H,T] (Falcon-1, 1A) or [B,H,T,dv] (Falcon-2, 2A), lam [B,H,T], S0 [B,H,dk,dv] or None,
    tail [B,H,dk] (the pending key k_pos) iff pos > 0. Returns (out [B,H,T,dv], S_final)."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    per_col = variant in (FALCON_2, FALCON_2A)
    inner = variant in (FALCON_1A, FALCON_2A)
    S = S0 if S0 is not None else torch.zeros(B, H, dk, dv, dtype=torch.float64)
    outs = []
    for t in range(T):
        tau = pos + t + 1
        if tau > 1:
            x = k[:, :, t - 1] if t > 0 else tail
            den = (x * x).sum(-1) + lam[:, :, t] + eps  # [B,H]
            nz = den != 0
            safe = torch.where(nz, den, torch.ones_like(den))
            b = beta[:, :, t]
            if per_col:
                eta = torch.where(nz[..., None], b / safe[..., None], torch.zeros_like(b))  # [B,H,dv]
                lm = lam[:, :, t][..., None]
            else:
                eta = torch.where(nz, b / safe, torch.zeros_like(b))  # [B,H]
                lm = lam[:, :, t]
            cap = 1.0 - eps_gamma
            raw = eta * lm
            alpha = torch.where(raw < cap, raw, torch.full_like(raw, cap))
            gamma = 1.0 - alpha
            y = v[:, :, t]
            r = y if inner else y - torch.einsum("bhkv,bhk->bhv", S, x)
            if per_col:
                S = gamma[..., None, :] * S + x[..., :, None] * (eta * r)[..., None, :]
            else:
                S = gamma[..., None, None] * S + eta[..., None, None] * x[..., :, None] * r[..., None, :]
        outs.append(torch.einsum("bhkv,bhk->bhv", S, q[:, :, t]))
    out = torch.stack(outs, dim=2) if outs else torch.zeros(B, H, 0, dv, dtype=torch.float64)
    return out, S


def _t(a):
    if a is None:
        return None
    if torch.is_tensor(a):
        return a.detach().cpu().double().clone()
    return torch.as_tensor(np.asarray(a, dtype=np.float64)).clone()


def falcon_ref_bwd(variant, q, k, v, beta, lam, dout, S0=None, dS_final=None, *, pos=0, tail=None,
                   eps=1e-6, eps_gamma=1e-6):
    """Gradients of sum(out * dout) + sum(S_final * dS_final) with respect to q, k, v, beta, lam,
    S0 and the tail key, as fp64 numpy arrays (dS0 / dtail are None when S0 / tail are None).
    `tail` may be given as [B,H,dk] or as the (keys [B,H,1,dk], vals) pair of the C oracle."""
    if isinstance(tail, (tuple, list)):
        tail = tail[0]
    if tail is not None:
        tail = _t(tail).reshape(q.shape[0], q.shape[1], -1)
    leaves = [_t(a).requires_grad_(True) for a in (q, k, v, beta, lam)]
    tS0 = _t(S0).requires_grad_(True) if S0 is not None else None
    ttail = tail.requires_grad_(True) if tail is not None else None
    out, S = forward_torch(variant, *leaves, tS0, pos=pos, tail=ttail, eps=eps, eps_gamma=eps_gamma)
    loss = (out * _t(dout)).sum()
    if dS_final is not None:
        loss = loss + (S * _t(dS_final)).sum()
    wrt = leaves + [a for a in (tS0, ttail) if a is not None]
    grads = torch.autograd.grad(loss, wrt, allow_unused=True) if loss.requires_grad else [None] * len(wrt)
    res = [g.numpy() if g is not None else np.zeros(tuple(a.shape)) for g, a in zip(grads, wrt)]
    names = ["dq", "dk", "dv", "dbeta", "dlam"]
    d = dict(zip(names, res[:5]))
    rest = res[5:]
    d["dS0"] = rest.pop(0) if tS0 is not None else None
    d["dtail"] = rest.pop(0) if ttail is not None else None
    return d
