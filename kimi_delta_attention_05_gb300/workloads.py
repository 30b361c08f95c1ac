"""Seeded synthetic workloads for the KDA forward pass.

This module only draws random numbers; it holds none of the method's
arithmetic.  It is the one piece shared by the oracle side (tests, CPU
baseline) and the CUDA side (tests, benchmark), so that both see the same
inputs.

Every workload is drawn on the CPU from ``torch.Generator().manual_seed(seed)``
in a fixed order -- [sequence lengths (packed varlen only)], q, k, v, g, beta,
A_log, dt_bias, initial_state -- then cast to the storage dtypes of the
flashkda.fwd parameter table (FlashKDA page, "Core Kernel API"): bf16 q, k, v,
g and beta logits; fp32 A_log [H] and dt_bias [H, K]; fp32 or bf16 states
[N, H, V, K]; int64 cu_seqlens [N+1].  N(m, s) below means mean m and
standard deviation s.
"""
from __future__ import annotations

import dataclasses
import math

import torch

HEAD_DIM = 128  # K = V = 128 (flashkda.fwd constraints: K == V == 128)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int                       # per-row length (dense) or packed total (varlen)
    H: int
    gate: str                    # "safe" | "unsafe"
    lower_bound: float
    qk_l2norm: bool
    qk_std: float
    g_std: float
    beta_std: float
    a_log_range: tuple           # A_log = log(U[lo, hi])
    init_state: str | None       # None | "f32" | "bf16"
    final_state: str | None      # None | "f32" | "bf16"
    n_seqs: int = 0              # >0: packed varlen with this many sequences
    max_len: int = 0             # varlen lengths ~ U{1..max_len}
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(HEAD_DIM)


WORKLOADS = {
    # tiny: one head, one chunk; parity only
    "tiny": Workload("tiny", 1, 64, 1, "safe", -5.0, True, 1.0, 1.0, 1.0, (1.0, 16.0),
                     None, "f32"),
    # dense batch with fp32 initial and final states
    "dense_batch": Workload("dense_batch", 4, 2048, 16, "safe", -5.0, True, 1.0, 1.0, 1.0,
                            (1.0, 16.0), "f32", "f32"),
    # long context, unsafe (softplus) gate, no states
    "long_context": Workload("long_context", 1, 8192, 32, "unsafe", -5.0, True, 1.0, 1.0, 1.0,
                             (1.0, 16.0), None, None),
    # 64 packed sequences, lengths U{1..4096}, per-sequence fp32 states
    "packed_varlen": Workload("packed_varlen", 1, 0, 16, "safe", -5.0, True, 1.0, 1.0, 1.0,
                              (1.0, 16.0), "f32", "f32", n_seqs=64, max_len=4096),
    # one long sequence with few heads (distributions as long_context, fp32 final
    # state): few sequence-heads for the GPU, so the state stage's chain is cut
    # into segments (the sequence split)
    "long_sequence": Workload("long_sequence", 1, 65536, 4, "unsafe", -5.0, True, 1.0, 1.0, 1.0,
                              (1.0, 16.0), None, "f32"),
    # numerical extremes: wide gate/beta logits, extreme A_log, no L2 norm, bf16 states
    "extremes": Workload("extremes", 2, 32768, 8, "safe", -5.0, False, 0.05, 4.0, 4.0,
                         (0.01, 64.0), "bf16", "bf16"),
    # decoding step (token-by-token path): 256 sequences x 1 token x 32 heads,
    # fp32 states carried from call to call (distributions as dense_batch)
    "decode": Workload("decode", 256, 1, 32, "safe", -5.0, True, 1.0, 1.0, 1.0, (1.0, 16.0),
                       "f32", "f32"),
}

# The chunked-path workloads in the order they are usually listed.
WORKLOAD_ORDER = ["tiny", "dense_batch", "long_context", "packed_varlen", "extremes", "long_sequence"]


def make_inputs(w: Workload, *, seed: int | None = None, lengths=None, T: int | None = None,
                H: int | None = None, B: int | None = None):
    """Draw the inputs of a workload on the CPU.

    ``lengths`` / ``T`` / ``H`` / ``B`` override the workload's sizes (for
    reduced parity cases that keep its distributions).  Returns a dict of CPU
    tensors: q, k, v, g, beta (bf16), A_log, dt_bias (fp32), initial_state
    (fp32/bf16 or None), cu_seqlens (int64 or None), plus the scalar
    arguments scale, lower_bound, gate, qk_l2norm, final_state dtype and N.
    """
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    K = V = HEAD_DIM
    Hh = w.H if H is None else H
    cu = None
    if w.n_seqs or lengths is not None:
        if lengths is None:
            lengths = torch.randint(1, w.max_len + 1, (w.n_seqs,), generator=gen)
        lengths = torch.as_tensor(lengths, dtype=torch.int64)
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(lengths, 0)
        Bb, Tt, N = 1, int(cu[-1]), len(lengths)
    else:
        Bb = w.B if B is None else B
        Tt = w.T if T is None else T
        N = Bb

    def normal(shape, std):
        return torch.randn(shape, generator=gen, dtype=torch.float32) * std

    q = normal((Bb, Tt, Hh, K), w.qk_std).to(torch.bfloat16)
    k = normal((Bb, Tt, Hh, K), w.qk_std).to(torch.bfloat16)
    v = normal((Bb, Tt, Hh, V), 1.0).to(torch.bfloat16)
    g = normal((Bb, Tt, Hh, K), w.g_std).to(torch.bfloat16)
    beta = normal((Bb, Tt, Hh), w.beta_std).to(torch.bfloat16)
    lo, hi = w.a_log_range
    A_log = torch.log(lo + (hi - lo) * torch.rand((Hh,), generator=gen, dtype=torch.float32))
    dt_bias = normal((Hh, K), 0.1)
    init = None
    if w.init_state is not None:
        init = normal((N, Hh, V, K), 0.1)
        if w.init_state == "bf16":
            init = init.to(torch.bfloat16)
    return dict(q=q, k=k, v=v, g=g, beta=beta, A_log=A_log, dt_bias=dt_bias,
                initial_state=init, cu_seqlens=cu, scale=w.scale, lower_bound=w.lower_bound,
                gate=w.gate, qk_l2norm=w.qk_l2norm, final_state=w.final_state, N=N)


def token_count(inputs) -> int:
    q = inputs["q"]
    return int(q.shape[0] * q.shape[1])
