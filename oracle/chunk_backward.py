"""Gradients of the KDA forward pass in chunked (WY / UT) form, fp64 numpy.

TEST INFRASTRUCTURE (see the package docstring).  A second, independent
statement of the backward pass (the "chunk_bwd" stage of the fla-kda code map,
fla-kda SKILL.md "Code map"): reverse-mode differentiation of the chunk algebra
that ``chunk_form.py`` writes out, taken by hand, step by step, instead of by
autograd over the token recurrence (``backward.py``).  It is pinned to that
autograd oracle (tests/test_backward_oracle.py) and exposes the per-chunk
gradient intermediates for debugging.

Per (sequence, head) and chunk of C tokens, with S the [V, K] state before the
chunk, x_hat the (optionally L2-normalised) q and k, Gamma the in-chunk
cumulative log decay, F_ij = exp(Gamma_i - Gamma_j) (per key channel, j <= i):

  G = strict_lower(sum_c k_ic k_jc F_ijc),  P = lower(sum_c q_ic k_jc F_ijc)
  M = I + Diag(beta) G,  T = M^-1 Diag(beta)
  Qg = q e^Gamma,  Kg = k e^Gamma,  Khat = k e^{Gamma_C - Gamma},  gC = e^{Gamma_C}
  W = T Kg,  U = T V,  Unew = U - W S^T
  O = scale (Qg S^T + P Unew),  S_C = S Diag(gC) + Unew^T Khat

The reverse pass walks the chunks last to first carrying dS = dL/dS_C:

  dU  = scale P^T dO + Khat dS^T         dS_prev = scale dO^T Qg + dS Diag(gC) - dU^T W
  dQg = scale dO S,  dP = lower(scale dO Unew^T),  dKhat = Unew dS,  dgC = colsum(S * dS)
  dW  = -dU S,  dV = T^T dU,  dKg = T^T dW,  dT = lower(dU V^T + dW Kg^T)
  dbeta = diag(M^-T dT) + rowsum(dA * G),  dA = strict_lower(-M^-T (dT Diag(beta)) M^-T)
  dG  = Diag(beta) dA

then through the pairwise sums G and P (each term's derivative with respect
to k, q and Gamma), the scalings, Gamma_t = sum_{s <= t} a_s, the gate
a = f(g + dt_bias), the L2 norm and the sigmoid of beta.  Every exponent is
<= 0, so no offset is needed in fp64; the inverse is numpy's (a library step).
"""
from __future__ import annotations

import numpy as np

from .recurrence import gate_activation


def _np64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()  # exact for bf16, fp32 and fp64
    return np.asarray(x, dtype=np.float64)


def _sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def gate_derivatives(z, A_log_h, gate: str, lower_bound: float):
    """da/dz and da/dA_log of the activated log decay a = gate(z) (fla-kda
    SKILL.md, "Gate contracts"): safe a = lb sigmoid(m z), m = exp(A_log) (1
    without A_log); unsafe a = -m softplus(z); logspace a = z."""
    z = np.asarray(z, dtype=np.float64)
    if gate == "logspace":
        return np.ones_like(z), np.zeros_like(z)
    m = 1.0 if A_log_h is None else float(np.exp(A_log_h))
    if gate == "unsafe":
        a = gate_activation(z, A_log_h, gate, lower_bound)
        return -m * _sigmoid(z), a
    s = _sigmoid(m * z)
    ds = s * (1.0 - s)
    return lower_bound * ds * m, lower_bound * ds * m * z


def chunk_backward(q, k, v, g, beta, dout, *, scale, A_log=None, dt_bias=None, lower_bound=-5.0,
                   gate="safe", beta_prob=False, qk_l2norm=False, l2_eps=1e-6, initial_state=None,
                   dfinal=None, cu_seqlens=None, chunk=64, keep=False):
    """Same arguments and result dict as ``kda_backward`` (gradients of
    <out, dout> + <final, dfinal> for q, k, v, g, beta, A_log, dt_bias and
    initial_state; None for an input given as None, and for A_log / dt_bias
    with the logspace gate).  ``keep=True`` adds "chunks": {(n, h): [per-chunk
    dicts of dS_end, dU, dQg, dP, dKhat, dW, dT, dGamma]}."""
    q, k, v, g, beta, dout = (_np64(x) for x in (q, k, v, g, beta, dout))
    A_log, dt_bias, init, dfin = _np64(A_log), _np64(dt_bias), _np64(initial_state), _np64(dfinal)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is not None:
        cu = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    else:
        cu = [b * T for b in range(B + 1)]
    N = len(cu) - 1
    R = B * T
    qf, kf, vf = q.reshape(R, H, K), k.reshape(R, H, K), v.reshape(R, H, V)
    gf, bf, of = g.reshape(R, H, K), beta.reshape(R, H), dout.reshape(R, H, V)
    dq, dk, dg = np.zeros((R, H, K)), np.zeros((R, H, K)), np.zeros((R, H, K))
    dv, dbeta = np.zeros((R, H, V)), np.zeros((R, H))
    dA_log, ddt_bias = np.zeros(H), np.zeros((H, K))
    dinit = np.zeros((N, H, V, K))
    kept = {}
    uses_params = gate != "logspace"
    for n in range(N):
        for h in range(H):
            Ah = None if A_log is None else A_log[h]
            bias = dt_bias[h] if (dt_bias is not None and uses_params) else np.zeros(K)
            S = np.zeros((V, K)) if init is None else init[n, h].copy()
            fwd = []
            for c0 in range(cu[n], cu[n + 1], chunk):       # forward: chunk quantities and S
                c1 = min(c0 + chunk, cu[n + 1])
                L = c1 - c0
                Q, Kc, Vc = qf[c0:c1, h], kf[c0:c1, h], vf[c0:c1, h]
                rq = 1.0 / np.sqrt((Q * Q).sum(-1, keepdims=True) + l2_eps) if qk_l2norm else np.ones((L, 1))
                rk = 1.0 / np.sqrt((Kc * Kc).sum(-1, keepdims=True) + l2_eps) if qk_l2norm else np.ones((L, 1))
                Qh, Kh = Q * rq, Kc * rk
                z = gf[c0:c1, h] + bias
                a = gate_activation(z, Ah, gate, lower_bound)
                b = bf[c0:c1, h] if beta_prob else _sigmoid(bf[c0:c1, h])
                Gam = np.cumsum(a, axis=0)
                low = np.tril(np.ones((L, L), dtype=bool))
                diff = np.where(low[:, :, None], Gam[:, None, :] - Gam[None, :, :], 0.0)
                F = np.where(low[:, :, None], np.exp(diff), 0.0)   # F_ijc, j <= i
                Gm = np.tril(np.einsum("ic,jc,ijc->ij", Kh, Kh, F), -1)
                P = np.einsum("ic,jc,ijc->ij", Qh, Kh, F)
                Minv = np.linalg.inv(np.eye(L) + b[:, None] * Gm)
                Tm = Minv * b[None, :]
                eG = np.exp(Gam)
                Qg, Kg = Qh * eG, Kh * eG
                Khat = Kh * np.exp(Gam[-1][None, :] - Gam)
                gC = eG[-1]
                W, U = Tm @ Kg, Tm @ Vc
                Unew = U - W @ S.T
                fwd.append(dict(c0=c0, c1=c1, Q=Q, Kc=Kc, Vc=Vc, Qh=Qh, Kh=Kh, rq=rq, rk=rk, z=z, b=b,
                                F=F, G=Gm, P=P, Minv=Minv, T=Tm, Qg=Qg, Kg=Kg, Khat=Khat, gC=gC, W=W,
                                Unew=Unew, S=S.copy(), eG=eG, Gam=Gam))
                S = S * gC[None, :] + Unew.T @ Khat
            dS = np.zeros((V, K)) if dfin is None else dfin[n, h].copy()
            chunks = []
            for c in reversed(fwd):                           # reverse over chunks
                c0, c1 = c["c0"], c["c1"]
                dO = of[c0:c1, h]
                S0, b = c["S"], c["b"]
                dU = scale * c["P"].T @ dO + c["Khat"] @ dS.T
                dQg = scale * dO @ S0
                dP = np.tril(scale * dO @ c["Unew"].T)
                dKhat = c["Unew"] @ dS
                dgC = (S0 * dS).sum(0)
                dW = -dU @ S0
                dT = np.tril(dU @ c["Vc"].T + dW @ c["Kg"].T)
                dv[c0:c1, h] = c["T"].T @ dU
                dKg = c["T"].T @ dW
                Minv = c["Minv"]
                db = np.einsum("ji,ji->i", Minv, dT)           # T = Minv Diag(beta)
                dA = np.tril(-Minv.T @ (dT * b[None, :]) @ Minv.T, -1)
                db += (dA * c["G"]).sum(1)                      # M = I + Diag(beta) G
                dG = dA * b[:, None]
                Kh, Qh, F = c["Kh"], c["Qh"], c["F"]
                # pairwise sums: each term's derivative with respect to k, q and Gamma
                dKh = np.einsum("ij,jc,ijc->ic", dG, Kh, F) + np.einsum("ij,ic,ijc->jc", dG, Kh, F)
                dQh = np.einsum("ij,jc,ijc->ic", dP, Kh, F)
                dKh += np.einsum("ij,ic,ijc->jc", dP, Qh, F)
                tG = np.einsum("ij,ic,jc,ijc->ijc", dG, Kh, Kh, F)
                tP = np.einsum("ij,ic,jc,ijc->ijc", dP, Qh, Kh, F)
                dGam = tG.sum(1) - tG.sum(0) + tP.sum(1) - tP.sum(0)
                # the scalings e^Gamma, e^{Gamma_C - Gamma}, e^{Gamma_C}
                eG, Gam = c["eG"], c["Gam"]
                dQh += dQg * eG
                dKh += dKg * eG + dKhat * np.exp(Gam[-1][None, :] - Gam)
                dGam += dQg * c["Qg"] + dKg * c["Kg"] - dKhat * c["Khat"]
                dGam[-1] += (dKhat * c["Khat"]).sum(0) + dgC * c["gC"]
                da = np.cumsum(dGam[::-1], axis=0)[::-1]        # Gamma_t = sum_{s <= t} a_s
                dadz, dadA = gate_derivatives(c["z"], Ah, gate, lower_bound)
                dz = da * dadz
                dg[c0:c1, h] = dz
                if uses_params:
                    ddt_bias[h] += dz.sum(0)
                    dA_log[h] += (da * dadA).sum()
                if qk_l2norm:   # x_hat = x r, r = (|x|^2 + eps)^-1/2: dx = r (dx_hat - x_hat (x_hat . dx_hat))
                    dq[c0:c1, h] = c["rq"] * (dQh - Qh * (Qh * dQh).sum(-1, keepdims=True))
                    dk[c0:c1, h] = c["rk"] * (dKh - Kh * (Kh * dKh).sum(-1, keepdims=True))
                else:
                    dq[c0:c1, h], dk[c0:c1, h] = dQh, dKh
                dbeta[c0:c1, h] = db if beta_prob else db * b * (1.0 - b)
                if keep:
                    chunks.append(dict(dS_end=dS.copy(), dU=dU, dQg=dQg, dP=dP, dKhat=dKhat, dW=dW,
                                       dT=dT, dGamma=dGam))
                dS = scale * dO.T @ c["Qg"] + dS * c["gC"][None, :] - dU.T @ c["W"]
            dinit[n, h] = dS
            if keep:
                kept[(n, h)] = chunks[::-1]
    out = {"q": dq.reshape(q.shape), "k": dk.reshape(k.shape), "v": dv.reshape(v.shape),
           "g": dg.reshape(g.shape), "beta": dbeta.reshape(beta.shape),
           "A_log": dA_log if (uses_params and A_log is not None) else None,
           "dt_bias": ddt_bias if (uses_params and dt_bias is not None) else None,
           "initial_state": dinit if init is not None else None}
    if keep:
        out["chunks"] = kept
    return out
