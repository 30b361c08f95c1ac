"""Gradients of the KDA forward pass in fp64: reverse-mode differentiation of a
plain token recurrence written with PyTorch CPU operations.

TEST INFRASTRUCTURE (see the package docstring): only tests, smoke() and the
benchmark's baseline legs use this module.

The forward here restates the recurrence of ``kda_oracle.c`` token by token
(fla-kda SKILL.md, "Gate contracts" for the gate forms; the KDA recurrence:
decay first, then the delta write with the decayed state, read-out after the
write):

    a_t = gate(g_t + dt_bias[h])            per key channel
    S   = S Diag(exp(a_t))
    S   = S + beta_t (v_t - S k_t) k_t^T     beta_t = sigmoid(beta logit)
    o_t = scale S q_t

with q, k optionally divided by sqrt(|x|^2 + eps).  The backward pass of the
"chunk_bwd" stage of the fla-kda code map computes the gradients of a loss
L = <out, dout> + <final_state, dfinal> with respect to every input; here they
come from autograd over this forward (a library step, like a matmul), in
fp64.  The forward is pinned to the C oracle and the gradients to central
finite differences (tests/test_backward_oracle.py).
"""
from __future__ import annotations

import numpy as np
import torch


def _t64(x, requires_grad=False):
    if x is None:
        return None
    if not torch.is_tensor(x):
        x = torch.as_tensor(np.asarray(x))
    x = x.detach().to("cpu", torch.float64).clone()
    x.requires_grad_(requires_grad)
    return x


def gate_torch(z, A_log_h, gate: str, lower_bound: float):
    """Activated log decay a of the pre-activation z (fp64 torch).  safe:
    lower_bound * sigmoid(exp(A_log) z) (A_log None -> multiplier 1); unsafe:
    -exp(A_log) softplus(z), softplus in the exact form max(z, 0) +
    log1p(exp(-|z|)); logspace: z is already a."""
    if gate == "logspace":
        return z
    if gate == "safe":
        m = 1.0 if A_log_h is None else torch.exp(A_log_h)
        return lower_bound * torch.sigmoid(m * z)
    if gate == "unsafe":
        sp = torch.clamp(z, min=0.0) + torch.log1p(torch.exp(-torch.abs(z)))
        return -torch.exp(A_log_h) * sp
    raise ValueError(gate)


def kda_forward_torch(q, k, v, g, beta, *, scale, A_log=None, dt_bias=None, lower_bound=-5.0,
                      gate="safe", beta_prob=False, qk_l2norm=False, l2_eps=1e-6,
                      initial_state=None, cu_seqlens=None):
    """Token recurrence on fp64 torch tensors (autograd-friendly).

    q, k, g: [B, T, H, K]; v: [B, T, H, V]; beta: [B, T, H]; A_log [H];
    dt_bias [H, K]; initial_state [N, H, V, K].  With cu_seqlens ([N+1]) B must
    be 1 and sequence n is rows cu[n]..cu[n+1].  Any K and V.  Returns
    (out [B, T, H, V], final [N, H, V, K])."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is not None:
        cu = [int(x) for x in (cu_seqlens.tolist() if torch.is_tensor(cu_seqlens) else cu_seqlens)]
        spans = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    else:
        spans = [(b, 0, T) for b in range(B)]
    N = len(spans)
    out_rows = [[None] * T for _ in range(B)]
    finals = []
    bmat = beta if beta_prob else torch.sigmoid(beta)
    for n, (b, t0, t1) in enumerate(spans):
        if initial_state is not None:
            S = initial_state[n]
        else:
            S = torch.zeros((H, V, K), dtype=torch.float64)
        for t in range(t0, t1):
            z = g[b, t] if gate == "logspace" else g[b, t] + (dt_bias if dt_bias is not None else 0.0)
            a = torch.stack([gate_torch(z[h], None if A_log is None else A_log[h], gate, lower_bound)
                             for h in range(H)])                         # [H, K]
            qt, kt = q[b, t], k[b, t]                                    # [H, K]
            if qk_l2norm:
                qt = qt / torch.sqrt((qt * qt).sum(-1, keepdim=True) + l2_eps)
                kt = kt / torch.sqrt((kt * kt).sum(-1, keepdim=True) + l2_eps)
            S = S * torch.exp(a)[:, None, :]                             # decay (per key channel)
            pred = torch.einsum("hvk,hk->hv", S, kt)
            S = S + bmat[b, t][:, None, None] * torch.einsum("hv,hk->hvk", v[b, t] - pred, kt)
            out_rows[b][t] = scale * torch.einsum("hvk,hk->hv", S, qt)   # [H, V]
        finals.append(S)
    zero = torch.zeros((H, V), dtype=torch.float64)
    out = torch.stack([torch.stack([r if r is not None else zero for r in rows]) for rows in out_rows])
    return out, torch.stack(finals)


def kda_backward(q, k, v, g, beta, dout, *, scale, A_log=None, dt_bias=None, lower_bound=-5.0,
                 gate="safe", beta_prob=False, qk_l2norm=False, l2_eps=1e-6, initial_state=None,
                 dfinal=None, cu_seqlens=None):
    """Gradients of L = <out, dout> + <final_state, dfinal> (dfinal None: no
    final-state term) with respect to q, k, v, g, beta, A_log, dt_bias and
    initial_state, as fp64 numpy arrays in a dict (None for an input given as
    None; for the logspace gate A_log and dt_bias get None, being unused).  g
    and beta are the raw inputs (logits, or log decays / beta itself in the
    logspace / beta_prob modes)."""
    qq, kk, vv, gg, bb = (_t64(x, True) for x in (q, k, v, g, beta))
    uses_gate_params = gate != "logspace"
    al = _t64(A_log, uses_gate_params) if A_log is not None else None
    db = _t64(dt_bias, uses_gate_params) if dt_bias is not None else None
    init = _t64(initial_state, True) if initial_state is not None else None
    out, fin = kda_forward_torch(qq, kk, vv, gg, bb, scale=scale, A_log=al, dt_bias=db,
                                 lower_bound=lower_bound, gate=gate, beta_prob=beta_prob,
                                 qk_l2norm=qk_l2norm, l2_eps=l2_eps, initial_state=init,
                                 cu_seqlens=cu_seqlens)
    loss = (out * _t64(dout)).sum()
    if dfinal is not None:
        loss = loss + (fin * _t64(dfinal)).sum()
    loss.backward()

    def grad(x):
        if x is None or not x.requires_grad:
            return None
        return (x.grad if x.grad is not None else torch.zeros_like(x)).numpy()

    return {"q": grad(qq), "k": grad(kk), "v": grad(vv), "g": grad(gg), "beta": grad(bb),
            "A_log": grad(al), "dt_bias": grad(db), "initial_state": grad(init),
            "out": out.detach().numpy(), "final": fin.detach().numpy()}
