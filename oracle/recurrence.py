"""ctypes front end of the fp64 token-recurrence oracle (``kda_oracle.c``).

TEST INFRASTRUCTURE (see the package docstring).  ``build()`` compiles the C
file with gcc; building the checker is not using it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libkda_oracle.so")
_lib = None

GATE_SAFE = 1
GATE_UNSAFE = 2
GATE_LOGSPACE = 3


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libkda_oracle.so``."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        os.makedirs(_LIB_DIR, exist_ok=True)
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def configure(lib):
    """Declare the C signatures on a loaded oracle library."""
    P = ctypes.c_void_p
    lib.kda_oracle_fwd.restype = ctypes.c_int
    lib.kda_oracle_fwd.argtypes = [
        P, P, P, P, P, ctypes.c_double, P, P, ctypes.c_double, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_double, P, P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int64, P, ctypes.c_int64, ctypes.c_int]
    lib.kda_oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = configure(ctypes.CDLL(build()))
    return _lib


def max_threads() -> int:
    return int(_load().kda_oracle_max_threads())


def _f32(x):
    """Widen an input (numpy array or torch tensor, any float dtype) to a
    contiguous float32 numpy array.  bf16 -> fp32 is exact."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        import torch
        x = x.detach().to("cpu", torch.float32).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def gate_activation(z, A_log_h, gate: str, lower_bound: float):
    """fp64 gate activation on pre-biased logits z = g + dt_bias.

    fla-kda SKILL.md, "Gate contracts": with a lower bound the activation is
    lower_bound * sigmoid(exp(A_log) * z) (A_log omitted -> multiplier one);
    without one it is -exp(A_log) * softplus(z).  "logspace" is chunk_kda
    without the in-kernel gate: z (= g, no bias) is already the log decay.
    """
    z = np.asarray(z, dtype=np.float64)
    if gate == "logspace":
        return z
    if gate == "safe":
        m = 1.0 if A_log_h is None else np.exp(np.float64(A_log_h))
        x = m * z
        sig = np.where(x >= 0, 1.0 / (1.0 + np.exp(-np.abs(x))),
                       np.exp(-np.abs(x)) / (1.0 + np.exp(-np.abs(x))))
        return lower_bound * sig
    if gate == "unsafe":
        m = np.exp(np.float64(A_log_h))
        sp = np.maximum(z, 0.0) + np.log1p(np.exp(-np.abs(z)))
        return -m * sp
    raise ValueError(gate)


def kda_recurrence(q, k, v, g, beta, *, scale, A_log=None, dt_bias=None, lower_bound=-5.0,
                   gate="safe", beta_prob=False, qk_l2norm=False, l2_eps=1e-6,
                   initial_state=None, cu_seqlens=None, units=None, threads=0, want_final=True):
    """fp64 token recurrence.

    q, k, g: [B, T, H, K]; v: [B, T, H, V]; beta: [B, T, H] (logits, or beta
    itself with ``beta_prob``).  ``gate``: "safe", "unsafe" or "logspace" (g is
    the log decay; A_log and dt_bias unused).
    With ``cu_seqlens`` ([N+1] int64) B must be 1 and the sequences are the
    packed rows cu[n]..cu[n+1]; otherwise sequence n is batch row n.
    initial_state: [N, H, V, K] or None.  ``units``: optional list of n*H+h
    to compute (others are left as NaN).  Returns (out [B,T,H,V] float64,
    final [N,H,V,K] float64 or None).
    """
    lib = _load()
    qf, kf, vf, gf, bf = (_f32(x) for x in (q, k, v, g, beta))
    B, T, H, K = qf.shape
    V = vf.shape[-1]
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        N = len(cu) - 1
    else:
        N = B
        cu = np.arange(B + 1, dtype=np.int64) * T
    Al = _f32(A_log)
    db = _f32(dt_bias)
    init = _f32(initial_state)
    if init is not None and init.shape != (N, H, V, K):
        raise ValueError(f"initial_state shape {init.shape} != {(N, H, V, K)}")
    out = np.full((B, T, H, V), np.nan, dtype=np.float64)
    final = np.full((N, H, V, K), np.nan, dtype=np.float64) if want_final else None
    u = None if units is None else np.ascontiguousarray(np.asarray(units, dtype=np.int64))
    mode = {"safe": GATE_SAFE, "unsafe": GATE_UNSAFE, "logspace": GATE_LOGSPACE}[gate]
    rc = lib.kda_oracle_fwd(
        _ptr(qf), _ptr(kf), _ptr(vf), _ptr(gf), _ptr(bf), float(scale), _ptr(Al), _ptr(db),
        float(lower_bound), mode, int(bool(beta_prob)), int(bool(qk_l2norm)), float(l2_eps),
        _ptr(init), _ptr(out),
        _ptr(final), _ptr(cu), N, H, K, V, _ptr(u), 0 if u is None else len(u), int(threads))
    if rc != 0:
        raise ValueError("kda_oracle_fwd rejected its arguments")
    return out, final
