"""GPU tests of the host-buffer entry point (kda_fwd_host): inputs and outputs
in host memory, the library pipelines the copies with the kernels.

Dense inputs are split along the token axis with the state handed from piece
to piece in fp32, which must leave every bit of the result as kda_fwd gives
it; packed inputs are split between sequences.  Both are also checked against
the fp64 oracle with the usual tolerances (tests/kda_testlib.py).
"""
import ctypes

import numpy as np
import pytest
import torch

from kimi_delta_attention_05_gb300 import kda_fwd_host
from kimi_delta_attention_05_gb300.kda import host_device_bytes, make_args
from kimi_delta_attention_05_gb300.workloads import WORKLOADS, make_inputs
from tests import kda_testlib as tl

pytestmark = pytest.mark.gpu

PIECE_BYTES = 32 << 20  # input bytes a piece aims at (kda_host.cu)


def _run_host(inp, pinned=True):
    """kda_fwd_host on (pinned) CPU copies of ``inp``; NaN-poisoned outputs."""
    h = {k: ((v.pin_memory() if pinned else v.clone()) if torch.is_tensor(v) else v)
         for k, v in inp.items()}
    out = torch.full(h["v"].shape, float("nan"), dtype=h["v"].dtype)
    fin = None
    fdt = inp.get("final_state")
    if fdt is not None:
        dt = torch.bfloat16 if fdt == "bf16" else torch.float32
        fin = torch.full((inp["N"], h["q"].shape[2], 128, 128), float("nan"), dtype=dt)
    if pinned:
        out = out.pin_memory()
        fin = None if fin is None else fin.pin_memory()
    lb = inp["lower_bound"] if inp["gate"] == "safe" else None
    kda_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], inp["scale"], out, h["A_log"],
                 h["dt_bias"], lb, h["initial_state"], fin, h["cu_seqlens"],
                 qk_l2norm=inp["qk_l2norm"], gate=inp["gate"],
                 beta_prob=inp.get("beta_prob", False))
    torch.cuda.synchronize()
    o = out.float().numpy().astype(np.float64)
    f = None if fin is None else fin.float().numpy().astype(np.float64)
    return o, f


def _pieces_dense(inp):
    B, T, H, _ = inp["q"].shape
    total = B * T * H * 1026
    P = min(64, max(1, -(-total // max(PIECE_BYTES, -(-total // 64)))))
    span = -(-(-(-T // P)) // 64) * 64
    return -(-T // span)


def test_dense_long_sequence_split_is_bit_exact():
    """One long sequence (eight heads) in token-range pieces: identical to kda_fwd."""
    inp = make_inputs(WORKLOADS["long_context"], T=16384, H=8, seed=61)
    assert _pieces_dense(inp) >= 2
    o_h, _ = _run_host(inp)
    o_d, _ = tl.run_gpu(inp)
    assert np.array_equal(o_h, o_d)
    ro, _ = tl.run_oracle(inp)
    tl.check_out(o_h, ro, "host long sequence")


def test_dense_batch_bf16_states_split_is_bit_exact():
    """Three sequences, bf16 initial and final state, four pieces: the state is
    carried in fp32 between pieces, so the final bf16 state is kda_fwd's."""
    inp = make_inputs(WORKLOADS["extremes"], B=3, T=4096, H=8, seed=62)
    assert inp["final_state"] == "bf16" and inp["initial_state"].dtype == torch.bfloat16
    assert _pieces_dense(inp) == 4
    o_h, f_h = _run_host(inp)
    o_d, f_d = tl.run_gpu(inp)
    assert np.array_equal(o_h, o_d) and np.array_equal(f_h, f_d)
    ro, rf = tl.run_oracle(inp)
    tl.check_out(o_h, ro, "host bf16 states")
    tl.check_state(f_h, rf, "host bf16 states")


def test_packed_sequences_in_groups():
    """Packed sequences (some empty) cut into groups of whole sequences."""
    rng = np.random.default_rng(63)
    lengths = [int(x) for x in rng.integers(1, 3000, size=24)]
    lengths[3] = 0
    lengths[10] = 0
    inp = make_inputs(WORKLOADS["packed_varlen"], lengths=lengths, H=4, seed=63)
    assert sum(lengths) * 4 * 1026 > 3 * PIECE_BYTES  # several groups
    o_h, f_h = _run_host(inp)
    o_d, f_d = tl.run_gpu(inp)
    assert tl.rel_rms(o_h, o_d) < 1e-3 and tl.rel_rms(f_h, f_d) < 1e-4
    ro, rf = tl.run_oracle(inp)
    tl.check_out(o_h, ro, "host packed")
    tl.check_state(f_h, rf, "host packed")


def test_pageable_host_memory_same_result():
    inp = make_inputs(WORKLOADS["dense_batch"], B=2, T=300, H=3, seed=64)
    o_p, f_p = _run_host(inp, pinned=True)
    o_u, f_u = _run_host(inp, pinned=False)
    assert np.array_equal(o_p, o_u) and np.array_equal(f_p, f_u)
    ro, rf = tl.run_oracle(inp)
    tl.check_out(o_p, ro, "host small")
    tl.check_state(f_p, rf, "host small")


def test_empty_sequences_final_is_initial():
    """T = 0: no output rows, the final state is the initial state."""
    inp = make_inputs(WORKLOADS["dense_batch"], B=2, T=1, H=2, seed=65)
    for k in ("q", "k", "v", "g", "beta"):
        inp[k] = inp[k][:, :0].contiguous()
    _, f = _run_host(inp)
    assert np.array_equal(f, inp["initial_state"].double().numpy())
    _, f_d = tl.run_gpu(inp)  # kda_fwd on device tensors with no storage
    assert np.array_equal(f_d, inp["initial_state"].double().numpy())


def test_device_bytes_cover_the_device_path():
    """The host call needs at least the device copies of inputs and output."""
    inp = make_inputs(WORKLOADS["long_context"], T=8192, H=4, seed=66)
    out = torch.empty_like(inp["v"])
    a = make_args(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"], out,
                  inp["A_log"], inp["dt_bias"], None, None, None, None, qk_l2norm=True,
                  gate="unsafe")
    assert host_device_bytes(a) >= 5 * inp["q"].numel() * 2


@pytest.mark.parametrize("gate,beta_prob", [("logspace", True), ("unsafe", False)])
def test_flags_through_host_entry(gate, beta_prob):
    """Caller-gated g and beta given as beta, through the host-buffer entry:
    identical to kda_fwd on the same inputs, and within the oracle tolerance."""
    inp = make_inputs(WORKLOADS["dense_batch"], B=2, T=700, H=4, seed=67)
    inp["gate"] = gate
    if gate == "logspace":
        inp["g"] = (-(inp["g"].float().abs())).to(torch.bfloat16)
    if beta_prob:
        inp["beta"] = torch.sigmoid(inp["beta"].float()).to(torch.bfloat16)
        inp["beta_prob"] = True
    o_h, f_h = _run_host(inp)
    o_d, f_d = tl.run_gpu(inp)
    assert np.array_equal(o_h, o_d) and np.array_equal(f_h, f_d)
    ro, rf = tl.run_oracle(inp)
    tl.check_out(o_h, ro, f"host {gate}")
    tl.check_state(f_h, rf, f"host {gate}")


def test_packed_bf16_states_through_host_entry():
    """Packed sequences with bf16 initial and final states (per-group slices of
    the state tensors)."""
    rng = np.random.default_rng(68)
    lengths = [int(x) for x in rng.integers(1, 5000, size=12)]
    inp = make_inputs(WORKLOADS["packed_varlen"], lengths=lengths, H=8, seed=68)
    inp["initial_state"] = inp["initial_state"].to(torch.bfloat16)
    inp["final_state"] = "bf16"
    o_h, f_h = _run_host(inp)
    ro, rf = tl.run_oracle(inp)
    tl.check_out(o_h, ro, "host packed bf16")
    tl.check_state(f_h, rf, "host packed bf16")


def test_g_in_fp32_through_host_entry():
    """fp32 log decays through the host-buffer entry: dense pieces (2-D copies of
    512-byte g rows) and packed groups."""
    gen = torch.Generator().manual_seed(69)
    inp = make_inputs(WORKLOADS["dense_batch"], B=2, T=8192, H=4, seed=69)
    inp.update(g=-(torch.randn(inp["g"].shape, generator=gen)).abs(), gate="logspace")
    o_h, f_h = _run_host(inp)
    o_d, f_d = tl.run_gpu(inp)
    assert np.array_equal(o_h, o_d) and np.array_equal(f_h, f_d)
    lengths = [3000, 17, 5000, 64, 2500]
    inp = make_inputs(WORKLOADS["packed_varlen"], lengths=lengths, H=4, seed=70)
    inp.update(g=-(torch.randn(inp["g"].shape, generator=gen)).abs(), gate="logspace")
    o_h, f_h = _run_host(inp)
    ro, rf = tl.run_oracle(inp)
    tl.check_out(o_h, ro, "host fp32 g packed")
    tl.check_state(f_h, rf, "host fp32 g packed")


@pytest.mark.parametrize("gate,B,T,H", [("unsafe", 1, 16384, 8), ("safe", 2, 16500, 4)])
def test_host_pieces_match_one_pass(gate, B, T, H):
    """Few sequence-heads and sequences of at least 256 chunks: the host entry
    cuts the tokens into pieces whose state passes from piece to piece in
    fp32; kda_fwd runs the same problem in one pass, its state never leaving
    fp32 between chunks either: the results are identical."""
    inp = make_inputs(WORKLOADS["dense_batch"], B=B, T=T, H=H, seed=71)
    inp.update(gate=gate)
    d = tl.to_device(inp)
    a = make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], torch.empty_like(d["v"]),
                  d["A_log"], d["dt_bias"], inp["lower_bound"] if gate == "safe" else None,
                  d["initial_state"], None, None, inp["qk_l2norm"], gate)
    from kimi_delta_attention_05_gb300 import kda as K
    assert K.load_library().kda_fwd_launches(ctypes.byref(a)) == 2  # one pass
    o_h, f_h = _run_host(inp)
    o_d, f_d = tl.run_gpu(inp)
    assert np.array_equal(o_h, o_d) and np.array_equal(f_h, f_d)
    ro, rf = tl.run_oracle(inp)
    tl.check_out(o_d, ro, "one pass, 256 chunks")
    tl.check_state(f_d, rf, "one pass, 256 chunks")


def test_two_streams_at_once():
    """Two calls issued on two streams without ordering between them: each
    result equals the same call run alone."""
    cases = [make_inputs(WORKLOADS["long_context"], T=16384, H=8, seed=72),
             make_inputs(WORKLOADS["extremes"], B=1, T=16500, H=8, seed=73)]
    alone = [tl.run_gpu(inp) for inp in cases]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    devs, outs, fins = [], [], []
    for inp in cases:
        d = tl.to_device(inp)
        devs.append(d)
        outs.append(torch.full_like(d["v"], float("nan")))
        fdt = inp.get("final_state")
        fins.append(None if fdt is None else torch.full(
            (inp["N"], d["q"].shape[2], 128, 128), float("nan"), device="cuda",
            dtype=torch.bfloat16 if fdt == "bf16" else torch.float32))
    torch.cuda.synchronize()
    from kimi_delta_attention_05_gb300 import kda_fwd
    for rep in range(3):
        for inp, d, out, fin, s in zip(cases, devs, outs, fins, streams):
            lb = inp["lower_bound"] if inp["gate"] == "safe" else None
            kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], out, d["A_log"],
                    d["dt_bias"], lb, d["initial_state"], fin, d["cu_seqlens"],
                    qk_l2norm=inp["qk_l2norm"], gate=inp["gate"], stream=s)
    torch.cuda.synchronize()
    for (o_ref, f_ref), out, fin in zip(alone, outs, fins):
        assert np.array_equal(out.float().cpu().numpy().astype(np.float64), o_ref)
        if fin is not None:
            assert np.array_equal(fin.float().cpu().numpy().astype(np.float64), f_ref)
