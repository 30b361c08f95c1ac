"""GPU parity of the token-by-token path (kda_fwd_recurrent, the decoding
entry point) against the fp64 oracle, through the C ABI.

Same tolerances as the chunked path (tests/kda_testlib.py); this path keeps
the state in fp32 throughout, so its errors are far below them.
"""
import numpy as np
import pytest
import torch

from kimi_delta_attention_05_gb300 import kda_fwd_recurrent
from kimi_delta_attention_05_gb300.workloads import WORKLOADS, make_inputs
from tests import kda_testlib as tl

pytestmark = pytest.mark.gpu


def _run_recurrent(inp, in_place=False):
    d = tl.to_device(inp)
    out = torch.full_like(d["v"], float("nan"))
    fin = None
    fdt = inp.get("final_state")
    if in_place:
        fin = d["initial_state"]
    elif fdt is not None:
        dt = torch.bfloat16 if fdt == "bf16" else torch.float32
        fin = torch.full((inp["N"], d["q"].shape[2], 128, 128), float("nan"), dtype=dt, device="cuda")
    lb = inp["lower_bound"] if inp["gate"] == "safe" else None
    kda_fwd_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], out, d["A_log"],
                      d["dt_bias"], lb, d["initial_state"], fin, d["cu_seqlens"],
                      qk_l2norm=inp["qk_l2norm"], gate=inp["gate"],
                      beta_prob=inp.get("beta_prob", False))
    torch.cuda.synchronize()
    o = out.float().cpu().numpy().astype(np.float64)
    f = None if fin is None else fin.float().cpu().numpy().astype(np.float64)
    return o, f


def _check(inp, tag, in_place=False):
    o, f = _run_recurrent(inp, in_place)
    ro, rf = tl.run_oracle(inp)
    r = tl.check_out(o, ro, tag)
    if f is not None:
        tl.check_state(f, rf, tag)
    return o, f, r


def test_decode_batch_one_token():
    """64 sequences of one token each, fp32 initial and final state."""
    inp = make_inputs(WORKLOADS["dense_batch"], B=64, T=1, H=16, seed=31)
    inp["final_state"] = "f32"
    _, _, (r, _) = _check(inp, "decode T=1")
    # fp32 state: what remains is the bf16 rounding of the output (uniform
    # relative error of +-2^-9, RMS 2^-9 / sqrt(3) = 1.1e-3) and the approximate
    # exp2 / log2 of the gate
    assert r < 2.5e-3


@pytest.mark.parametrize("gate,beta_prob,l2", [
    ("safe", False, True), ("unsafe", False, True), ("logspace", False, False),
    ("safe", True, False), ("unsafe", True, True)])
def test_multi_token_modes(gate, beta_prob, l2):
    inp = make_inputs(WORKLOADS["dense_batch"], B=2, T=37, H=3, seed=32)
    inp.update(gate=gate, qk_l2norm=l2, final_state="f32")
    if gate == "logspace":
        inp["g"] = (-(inp["g"].float().abs())).to(torch.bfloat16)
    if beta_prob:
        inp["beta"] = torch.sigmoid(inp["beta"].float()).to(torch.bfloat16)
        inp["beta_prob"] = True
    _check(inp, f"recurrent {gate} beta_prob={beta_prob} l2={l2}")


@pytest.mark.parametrize("gate", ["logspace", "unsafe"])
def test_g_in_fp32(gate):
    inp = make_inputs(WORKLOADS["decode"], B=8, T=3, H=4, seed=36)
    gen = torch.Generator().manual_seed(37)
    g = torch.randn(inp["g"].shape, generator=gen) * 2.0
    if gate == "logspace":
        g = -g.abs()
    inp.update(g=g, gate=gate)
    _check(inp, f"recurrent fp32 g ({gate})")


def test_varlen_with_empty_sequences_in_place_state():
    """Packed sequences (two empty), the final state written over the initial
    state buffer."""
    inp = make_inputs(WORKLOADS["packed_varlen"], lengths=[3, 0, 1, 9, 0, 2], H=4, seed=33)
    inp["final_state"] = "f32"
    _check(inp, "recurrent varlen in place", in_place=True)


def test_bf16_states_extreme_inputs():
    inp = make_inputs(WORKLOADS["extremes"], B=3, T=5, H=4, seed=34)
    _check(inp, "recurrent bf16 states")


def test_matches_chunked_path():
    """The recurrent and the chunked path agree (both against the oracle)."""
    inp = make_inputs(WORKLOADS["dense_batch"], B=2, T=70, H=2, seed=35)
    inp["final_state"] = "f32"
    o1, f1, _ = _check(inp, "recurrent")
    o2, f2 = tl.run_gpu(inp)
    assert tl.rel_rms(o1, o2) < 5e-3 and tl.rel_rms(f1, f2) < 2e-3
