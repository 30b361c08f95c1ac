"""Sequence split inside one GPU: for very few sequence-heads the state
stage's chain is cut into segments.  The state after a segment is affine in
the state before it (S_end = S_start M + R), so one launch runs segment 0
beside each later segment's R (from a zero state) and M (from the identity,
U taken as zero), a small kernel chains the segment states, and a second
launch re-runs the later segments from them.

Checked against the fp64 oracle (outputs and final states, fp32 and bf16
states, ragged last chunk), against the unsplit pass of the host-buffer
entry (which never splits), and for the launch count that shows the split."""
import ctypes

import numpy as np
import pytest
import torch

from kimi_delta_attention_05_gb300 import kda as K
from kimi_delta_attention_05_gb300.workloads import WORKLOADS, make_inputs
from tests import kda_testlib as tl

pytestmark = pytest.mark.gpu


def _launches(inp):
    d = tl.to_device(inp)
    lb = inp["lower_bound"] if inp["gate"] == "safe" else None
    a = K.make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], torch.empty_like(d["v"]),
                    d["A_log"], d["dt_bias"], lb, d["initial_state"], None, None, inp["qk_l2norm"],
                    inp["gate"])
    return K.load_library().kda_fwd_launches(ctypes.byref(a))


def _host(inp):
    host = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in inp.items()}
    out = torch.full(inp["v"].shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    fin = None
    if inp.get("final_state") is not None:
        dt = torch.bfloat16 if inp["final_state"] == "bf16" else torch.float32
        fin = torch.full((inp["N"], inp["q"].shape[2], 128, 128), float("nan"), dtype=dt).pin_memory()
    lb = inp["lower_bound"] if inp["gate"] == "safe" else None
    K.kda_fwd_host(host["q"], host["k"], host["v"], host["g"], host["beta"], inp["scale"], out,
                   host["A_log"], host["dt_bias"], lb, host["initial_state"], fin, None,
                   qk_l2norm=inp["qk_l2norm"], gate=inp["gate"])
    torch.cuda.synchronize()
    return out.double().numpy(), None if fin is None else fin.double().numpy()


CASES = [
    # name, workload, overrides, final state dtype
    ("unsafe, no states", "long_context", dict(T=16384, H=2, seed=101), "f32"),
    ("safe, fp32 states, ragged", "dense_batch", dict(B=1, T=12300, H=3, seed=102), "f32"),
    ("extremes, bf16 states", "extremes", dict(B=1, T=16384, H=2, seed=103), "bf16"),
]


@pytest.mark.parametrize("name,workload,kw,fdt", CASES, ids=[c[0] for c in CASES])
def test_split_pass_matches_oracle_and_unsplit(name, workload, kw, fdt):
    inp = make_inputs(WORKLOADS[workload], **kw)
    inp["final_state"] = fdt
    assert _launches(inp) == 4  # chunk stage, state runs, segment chain, state re-runs
    o, f = tl.run_gpu(inp)
    ro, rf = tl.run_oracle(inp)
    tl.check_out(o, ro, name)
    tl.check_state(f, rf, name)
    o_u, f_u = _host(inp)  # the same problem without the split
    assert tl.rel_rms(o, o_u) < 3e-3 and tl.rel_rms(f, f_u) < 3e-3


def test_split_is_deterministic():
    inp = make_inputs(WORKLOADS["long_context"], T=16384, H=1, seed=104)
    inp["final_state"] = "f32"
    o1, f1 = tl.run_gpu(inp)
    o2, f2 = tl.run_gpu(inp)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(f1, f2)
