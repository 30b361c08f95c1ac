"""Helpers shared by the GPU parity tests: run the CUDA path and the oracle on
the same seeded inputs, and compare them with the stated tolerances.

Tolerances (rel-RMS = ||x - ref||_2 / ||ref||_2 over the whole tensor, the
relative-RMS style of the fla ``assert_close`` helper described in the
fla-correctness-coverage skill):
  out          : rel-RMS <= 5e-3 and max |x - ref| <= 2e-2 * max |ref|
  fp32 final   : rel-RMS <= 2e-3
  bf16 final   : rel-RMS <= 2e-3 (rounding the exact state to bf16 alone
                 costs about 1.1e-3 of it)
Every output element must be finite (outputs are NaN-poisoned before calls,
so a missed write shows up as NaN).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from kimi_delta_attention_05_gb300 import kda_fwd

OUT_RMS = 5e-3
OUT_MAXABS = 2e-2
STATE_RMS = 2e-3


def to_device(inp, device="cuda"):
    return {k: (v.to(device) if torch.is_tensor(v) else v) for k, v in inp.items()}


def run_gpu(inp, *, final=True, a_log=True, dt_bias=True, stream=None):
    """Run the CUDA path on device copies of ``inp`` with NaN-poisoned outputs.
    Returns (out float64 numpy, final float64 numpy or None)."""
    d = to_device(inp)
    out = torch.full_like(d["v"], float("nan"))
    fin = None
    fdt = inp.get("final_state")
    if final and fdt is not None:
        dt = torch.bfloat16 if fdt == "bf16" else torch.float32
        fin = torch.full((inp["N"], d["q"].shape[2], 128, 128), float("nan"), dtype=dt,
                         device="cuda")
    lb = inp["lower_bound"] if inp["gate"] == "safe" else None
    if stream is not None:  # the copies and NaN fills above ran on the current stream
        stream.wait_stream(torch.cuda.current_stream())
    kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], out,
            d["A_log"] if a_log else None, d["dt_bias"] if dt_bias else None, lb,
            d["initial_state"], fin, d["cu_seqlens"], qk_l2norm=inp["qk_l2norm"],
            gate=inp["gate"], beta_prob=inp.get("beta_prob", False), stream=stream)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy().astype(np.float64)
    f = None if fin is None else fin.float().cpu().numpy().astype(np.float64)
    return o, f


def run_oracle(inp, *, units=None, a_log=True, dt_bias=True):
    return oracle.kda_recurrence(
        inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], scale=inp["scale"],
        A_log=inp["A_log"] if a_log else None, dt_bias=inp["dt_bias"] if dt_bias else None,
        lower_bound=inp["lower_bound"], gate=inp["gate"], beta_prob=inp.get("beta_prob", False),
        qk_l2norm=inp["qk_l2norm"],
        initial_state=inp["initial_state"], cu_seqlens=inp["cu_seqlens"], units=units)


def rel_rms(x, ref):
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def check_out(o, ref, tag=""):
    assert np.isfinite(o).all(), f"{tag}: non-finite outputs (missed write or overflow)"
    r = rel_rms(o, ref)
    m = float(np.abs(o - ref).max()) if ref.size else 0.0
    bound = OUT_MAXABS * float(np.abs(ref).max()) if ref.size else 0.0
    assert r <= OUT_RMS, f"{tag}: out rel-RMS {r:.3e} > {OUT_RMS}"
    assert m <= bound + 1e-30, f"{tag}: out max-abs {m:.3e} > {bound:.3e}"
    return r, m


def check_state(f, ref, tag=""):
    assert np.isfinite(f).all(), f"{tag}: non-finite final state"
    r = rel_rms(f, ref)
    assert r <= STATE_RMS, f"{tag}: final-state rel-RMS {r:.3e} > {STATE_RMS}"
    return r


# Margins of the full-size parity checks, printed at the end of the session
# (tests/conftest.py, pytest_terminal_summary): (tag, out rel-RMS, out
# max-abs / max|ref|, worst unit's out rel-RMS, final-state rel-RMS or None).
MARGINS = []


def record_margin(tag, out_rms, out_maxabs_ratio, worst_unit_rms, state_rms):
    MARGINS.append((tag, out_rms, out_maxabs_ratio, worst_unit_rms, state_rms))


# Gradient errors of the backward-pass tests: (tag, {input name: rel-RMS}).
GRAD_MARGINS = []


def record_grad_margin(tag, errs):
    GRAD_MARGINS.append((tag, dict(errs)))


def unit_rows(inp, units):
    """Token rows [(b, t0, t1, h)] covered by (n*H + h) units."""
    H = inp["q"].shape[2]
    rows = []
    cu = inp["cu_seqlens"]
    T = inp["q"].shape[1]
    for u in units:
        n, h = divmod(int(u), H)
        if cu is not None:
            rows.append((0, int(cu[n]), int(cu[n + 1]), h))
        else:
            rows.append((n, 0, T, h))
    return rows


def compare_units(inp, o, f, units, tag=""):
    """Compare GPU results on a subset of (sequence, head) units with the oracle."""
    ro, rf = run_oracle(inp, units=units)
    xs, rs = [], []
    for (b, t0, t1, h) in unit_rows(inp, units):
        xs.append(o[b, t0:t1, h].ravel())
        rs.append(ro[b, t0:t1, h].ravel())
    res = {"out": check_out(np.concatenate(xs), np.concatenate(rs), tag)}
    if f is not None:
        H = inp["q"].shape[2]
        fx = np.stack([f[u // H, u % H] for u in units])
        fr = np.stack([rf[u // H, u % H] for u in units])
        res["state"] = check_state(fx, fr, tag)
    return res
