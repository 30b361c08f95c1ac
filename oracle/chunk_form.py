"""Chunked (WY / UT) form of the KDA forward pass, fp64 numpy, exact exponentials.

TEST INFRASTRUCTURE (see the package docstring).  A second, independent
restatement of the method, used (1) as a pinned cross-check of the token
recurrence and (2) to expose per-chunk intermediates so that each GPU stage
can be debugged against it.

Per sequence and head, the tokens are cut into chunks of C tokens; chunks
restart at every sequence start and the last one may be partial.  Inside a
chunk, with a_t the activated gate (natural log, per key channel):

  Gamma_i = sum_{s<=i} a_s                     in-chunk cumulative log-decay
  A_ij    = beta_i <k_i * exp(Gamma_i - Gamma_j), k_j>        (j <  i)
  P_ij    =        <q_i * exp(Gamma_i - Gamma_j), k_j>        (j <= i)
  T       = (I + A)^-1 Diag(beta)
  W       = T (K * exp(Gamma)),   U = T V
  U_new   = U - W S0^T
  O       = scale (Q * exp(Gamma)) S0^T + scale P U_new
  S_C     = S0 Diag(exp(Gamma_C)) + U_new^T (K * exp(Gamma_C - Gamma))

This is the algebra that the "gate.py" (gate + cumulative decay), "wy_fast.py"
(W, U recompute), "solve_tril" and "chunk_delta_h" / "chunk_o" (state and
output) stages of the fla-org/flash-linear-attention KDA code map compute
(fla-kda SKILL.md, "Code map"; chunk_o.py section: the forward adds the
inter- and intra-chunk parts).  It follows from the recurrence by unrolling
it over the chunk; every exponent here is <= 0, so no offset trick is needed
in fp64.  The triangular solve uses numpy's dense solver as a library step.
"""
from __future__ import annotations

import numpy as np

from .recurrence import gate_activation


def _np64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu", torch.float32).numpy()
    return np.asarray(x, dtype=np.float64)


def _sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def chunk_form(q, k, v, g, beta, *, scale, A_log=None, dt_bias=None, lower_bound=-5.0,
               gate="safe", beta_prob=False, qk_l2norm=False, l2_eps=1e-6, initial_state=None,
               cu_seqlens=None, chunk=64, units=None, keep=False):
    """Same arguments and return values as ``kda_recurrence``; with
    ``keep=True`` also returns a dict {(n, h): [per-chunk dicts]} holding
    Gamma, A, P, T, W, U, U_new, O, S0 and S_end for every chunk."""
    q, k, v, g, beta = (_np64(x) for x in (q, k, v, g, beta))
    A_log, dt_bias, init = _np64(A_log), _np64(dt_bias), _np64(initial_state)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is not None:
        cu = np.asarray(cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
                        dtype=np.int64)
        N = len(cu) - 1
    else:
        N = B
        cu = np.arange(B + 1, dtype=np.int64) * T
    qf = q.reshape(B * T, H, K)
    kf = k.reshape(B * T, H, K)
    vf = v.reshape(B * T, H, V)
    gf = g.reshape(B * T, H, K)
    bf = beta.reshape(B * T, H)
    out = np.full((B * T, H, V), np.nan)
    final = np.full((N, H, V, K), np.nan)
    kept = {}
    todo = range(N * H) if units is None else units
    for unit in todo:
        n, h = divmod(int(unit), H)
        S = np.zeros((V, K)) if init is None else init[n, h].copy()
        Ah = None if A_log is None else A_log[h]
        db = np.zeros(K) if (dt_bias is None or gate == "logspace") else dt_bias[h]
        chunks = []
        for c0 in range(cu[n], cu[n + 1], chunk):
            c1 = min(c0 + chunk, cu[n + 1])
            L = c1 - c0
            Qc, Kc, Vc = qf[c0:c1, h], kf[c0:c1, h], vf[c0:c1, h]
            if qk_l2norm:
                Qc = Qc / np.sqrt((Qc * Qc).sum(-1, keepdims=True) + l2_eps)
                Kc = Kc / np.sqrt((Kc * Kc).sum(-1, keepdims=True) + l2_eps)
            a = gate_activation(gf[c0:c1, h] + db, Ah, gate, lower_bound)
            b = bf[c0:c1, h] if beta_prob else _sigmoid(bf[c0:c1, h])
            Gam = np.cumsum(a, axis=0)                       # [L, K]
            diff = Gam[:, None, :] - Gam[None, :, :]         # Gamma_i - Gamma_j
            low = np.tril(np.ones((L, L), dtype=bool))       # j <= i
            F = np.where(low[:, :, None], np.exp(np.where(low[:, :, None], diff, 0.0)), 0.0)
            A = b[:, None] * np.einsum("ic,ijc,jc->ij", Kc, F, Kc)
            A = np.tril(A, -1)
            P = np.einsum("ic,ijc,jc->ij", Qc, F, Kc)
            Tm = np.linalg.solve(np.eye(L) + A, np.diag(b))
            eg = np.exp(Gam)
            W = Tm @ (Kc * eg)
            U = Tm @ Vc
            Unew = U - W @ S.T
            O = scale * ((Qc * eg) @ S.T + P @ Unew)
            Khat = Kc * np.exp(Gam[-1][None, :] - Gam)
            S_end = S * eg[-1][None, :] + Unew.T @ Khat
            out[c0:c1, h] = O
            if keep:
                chunks.append(dict(Gamma=Gam, A=A, P=P, T=Tm, W=W, U=U, U_new=Unew, O=O, S0=S,
                                   S_end=S_end, beta=b))
            S = S_end
        final[n, h] = S
        if keep:
            kept[(n, h)] = chunks
    out = out.reshape(B, T, H, V)
    return (out, final, kept) if keep else (out, final)
