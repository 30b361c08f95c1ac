"""GPU backward pass (kda_bwd) against the fp64 backward oracle.

Every gradient (q, k, v, g, beta, A_log, dt_bias, initial state) element by
element on small cases: every gate form, beta given or as logits, with and
without the L2 norm, g in bf16 or fp32, fp32 and bf16 initial states, a final-state gradient,
packed sequences including empty ones, ragged lengths across the
64-token chunks and their 16-token blocks, and many heads.  Tolerance (fp32
arithmetic from bf16 inputs): rel-RMS <= 1e-3 and max-abs <= 1e-2 max|ref| for
every gradient tensor.
"""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_05_gb300 import kda as K
from kimi_delta_attention_05_gb300.workloads import WORKLOADS, make_inputs
from tests import kda_testlib as tl

pytestmark = pytest.mark.gpu

GRAD_RMS = 1e-3
GRAD_MAXABS = 1e-2


def _check(name, x, ref):
    assert x.shape == ref.shape, (name, x.shape, ref.shape)
    assert np.isfinite(x).all(), name
    r = tl.rel_rms(x, ref)
    m = float(np.abs(x - ref).max()) if ref.size else 0.0
    bound = GRAD_MAXABS * float(np.abs(ref).max()) if ref.size else 0.0
    assert r <= GRAD_RMS, f"{name}: rel-RMS {r:.3e}"
    assert m <= bound + 1e-30, f"{name}: max-abs {m:.3e} > {bound:.3e}"
    return r


def _run(inp, dfinal=True, tag=""):
    gen = torch.Generator().manual_seed(123)
    dout = (torch.randn(inp["v"].shape, generator=gen) * 0.5).to(torch.bfloat16)
    H = inp["q"].shape[2]
    dfin = torch.randn((inp["N"], H, 128, 128), generator=gen) * 0.1 if dfinal else None
    d = tl.to_device(inp)
    lb = inp["lower_bound"] if inp["gate"] == "safe" else None
    grads = K.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], dout.cuda(), d["A_log"],
                      d["dt_bias"], lb, d["initial_state"], None if dfin is None else dfin.cuda(),
                      d["cu_seqlens"], qk_l2norm=inp["qk_l2norm"], gate=inp["gate"],
                      beta_prob=inp.get("beta_prob", False))
    torch.cuda.synchronize()
    ref = oracle.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout.double().numpy(),
                              scale=inp["scale"], A_log=inp["A_log"], dt_bias=inp["dt_bias"],
                              lower_bound=inp["lower_bound"], gate=inp["gate"],
                              beta_prob=inp.get("beta_prob", False), qk_l2norm=inp["qk_l2norm"],
                              initial_state=inp["initial_state"],
                              dfinal=None if dfin is None else dfin.double().numpy(),
                              cu_seqlens=inp["cu_seqlens"])
    errs = {}
    for name in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state"):
        if ref[name] is None:
            assert grads.get(name) is None, name
            continue
        errs[name] = _check(f"{tag} d{name}", grads[name].double().cpu().numpy(), ref[name])
    tl.record_grad_margin(tag, errs)
    return errs


@pytest.mark.parametrize("T", [1, 7, 8, 9, 15, 16, 17, 64, 130])
def test_backward_dense_safe(T):
    inp = make_inputs(WORKLOADS["dense_batch"], B=2, T=T, H=2, seed=200 + T)
    _run(inp, tag=f"safe T={T}")


def test_backward_unsafe_no_states():
    inp = make_inputs(WORKLOADS["long_context"], T=150, H=2, seed=210)
    _run(inp, dfinal=False, tag="unsafe")


def test_backward_unsafe_final_only():
    inp = make_inputs(WORKLOADS["long_context"], T=70, H=3, seed=211)
    _run(inp, dfinal=True, tag="unsafe dfinal")


def test_backward_extremes_bf16_state_no_l2():
    inp = make_inputs(WORKLOADS["extremes"], B=1, T=120, H=2, seed=212)
    _run(inp, tag="extremes")


def test_backward_logspace_beta_given():
    inp = make_inputs(WORKLOADS["dense_batch"], B=1, T=90, H=2, seed=213)
    gen = torch.Generator().manual_seed(214)
    inp["g"] = (-(torch.randn(inp["g"].shape, generator=gen)).abs()).to(torch.bfloat16)
    inp["beta"] = torch.sigmoid(inp["beta"].float()).to(torch.bfloat16)
    inp.update(gate="logspace", beta_prob=True)
    _run(inp, tag="logspace")


@pytest.mark.parametrize("gate", ["logspace", "unsafe"])
def test_backward_g_in_fp32(gate):
    """g given in fp32 (KDA_G_FP32): the log decays themselves (logspace) or
    unsafe-gate logits, read without a bf16 rounding."""
    inp = make_inputs(WORKLOADS["long_context"], T=150, H=2, seed=250)
    gen = torch.Generator().manual_seed(251)
    if gate == "logspace":
        inp["g"] = -(torch.rand(inp["g"].shape, generator=gen, dtype=torch.float32) * 0.3 + 1e-3)
        inp.update(gate="logspace")
    else:
        inp["g"] = torch.randn(inp["g"].shape, generator=gen, dtype=torch.float32) * 2.0
    _run(inp, tag=f"g fp32 {gate}")


def test_backward_packed_with_empty_sequences():
    inp = make_inputs(WORKLOADS["packed_varlen"], lengths=[17, 0, 1, 40, 16], H=2, seed=215)
    _run(inp, tag="packed")


def test_backward_safe_without_a_log():
    inp = make_inputs(WORKLOADS["dense_batch"], B=1, T=33, H=2, seed=216)
    inp["A_log"] = None
    _run(inp, tag="no A_log")


def test_backward_no_tokens():
    """T = 0 (dense, two sequences with states): no chunk runs; the
    initial-state gradient is dfinal and the A_log / dt_bias sums are zero."""
    H = 3
    gen = torch.Generator().manual_seed(260)
    e = lambda *sh: torch.empty(sh, dtype=torch.bfloat16, device="cuda")
    q, k, v, g = e(2, 0, H, 128), e(2, 0, H, 128), e(2, 0, H, 128), e(2, 0, H, 128)
    beta = e(2, 0, H)
    A_log = torch.rand(H, generator=gen).cuda()
    dt_bias = torch.randn((H, 128), generator=gen).cuda()
    init = torch.randn((2, H, 128, 128), generator=gen).cuda()
    dfin = torch.randn((2, H, 128, 128), generator=gen).cuda()
    grads = K.kda_bwd(q, k, v, g, beta, 0.1, e(2, 0, H, 128), A_log, dt_bias, -5.0, init, dfin, None,
                      qk_l2norm=True, gate="safe")
    torch.cuda.synchronize()
    assert torch.equal(grads["initial_state"], dfin)
    assert torch.count_nonzero(grads["A_log"]) == 0 and torch.count_nonzero(grads["dt_bias"]) == 0


def test_backward_rejects_bad_arguments():
    lib = K.load_library()
    a = K.kda_bwd_args()
    assert lib.kda_bwd(None, None, 0, None) == 1
    assert lib.kda_bwd_workspace_bytes(None) == 0
    import ctypes
    assert lib.kda_bwd(ctypes.byref(a), None, 0, None) != 0  # K = V = 0, flags 0


ITEM_BYTES = 559872  # workspace per (64-token chunk slot, head)


@pytest.mark.parametrize("H", [24, 160])
def test_backward_many_heads(H):
    """Many (chunk, head) items per launch, checked against the oracle; the
    workspace is one item per chunk slot and head."""
    inp = make_inputs(WORKLOADS["dense_batch"], B=1, T=70, H=H, seed=220 + H)
    d = tl.to_device(inp)
    a, _ = K.make_bwd_args(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"],
                           torch.empty_like(d["v"]), d["A_log"], d["dt_bias"], inp["lower_bound"],
                           d["initial_state"], None, None, qk_l2norm=True, gate="safe")
    assert K.bwd_workspace_bytes(a) == 2 * H * ITEM_BYTES
    _run(inp, tag=f"H={H}")


def test_backward_packed_workspace():
    """Packed sequences: a 256-byte header for the chunk prefix, then one item
    per chunk slot (ceil(T / 64) + N slots) and head."""
    inp = make_inputs(WORKLOADS["packed_varlen"], lengths=[17, 0, 1, 40, 16], H=2, seed=230)
    d = tl.to_device(inp)
    a, _ = K.make_bwd_args(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"],
                           torch.empty_like(d["v"]), d["A_log"], d["dt_bias"], inp["lower_bound"],
                           d["initial_state"], None, d["cu_seqlens"], qk_l2norm=True, gate="safe")
    T, N = 74, 5
    assert K.bwd_workspace_bytes(a) == 256 + ((T + 63) // 64 + N) * 2 * ITEM_BYTES


def _head_slice(inp, h, dout, dfin):
    """Inputs of head h alone (heads are independent), for the oracle."""
    s3 = lambda x: None if x is None else x[:, :, h:h + 1]
    st = lambda x: None if x is None else x[:, h:h + 1]
    return dict(q=s3(inp["q"]), k=s3(inp["k"]), v=s3(inp["v"]), g=s3(inp["g"]), beta=inp["beta"][:, :, h:h + 1],
                dout=dout[:, :, h:h + 1], A_log=inp["A_log"][h:h + 1], dt_bias=inp["dt_bias"][h:h + 1],
                initial_state=st(inp["initial_state"]), dfinal=None if dfin is None else st(dfin),
                cu_seqlens=inp["cu_seqlens"])


@pytest.mark.parametrize("workload,heads", [("long_context", (0, 29)), ("dense_batch", (5,)), ("extremes", (6,))])
def test_backward_full_size_sampled(workload, heads):
    """The full-size workload through kda_bwd (every chunk of every head, the
    launch configuration the benchmark times), checked against the chunked fp64
    oracle on sampled heads: every token gradient of the head, its dA_log and
    dt_bias sums and (with states) its initial-state gradient."""
    inp = make_inputs(WORKLOADS[workload])
    gen = torch.Generator().manual_seed(77)
    dout = (torch.randn(inp["v"].shape, generator=gen) * 0.5).to(torch.bfloat16)
    H = inp["q"].shape[2]
    dfin = torch.randn((inp["N"], H, 128, 128), generator=gen) * 0.1 if inp["initial_state"] is not None else None
    d = tl.to_device(inp)
    lb = inp["lower_bound"] if inp["gate"] == "safe" else None
    grads = K.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], dout.cuda(), d["A_log"],
                      d["dt_bias"], lb, d["initial_state"], None if dfin is None else dfin.cuda(),
                      d["cu_seqlens"], qk_l2norm=inp["qk_l2norm"], gate=inp["gate"])
    torch.cuda.synchronize()
    del d  # the extremes workload's 4.6 GB workspace is freed with the call; inputs go too
    for h in heads:
        a = _head_slice(inp, h, dout, dfin)
        ref = oracle.chunk_backward(a["q"], a["k"], a["v"], a["g"], a["beta"], a["dout"], scale=inp["scale"],
                                    A_log=a["A_log"], dt_bias=a["dt_bias"], lower_bound=inp["lower_bound"],
                                    gate=inp["gate"], qk_l2norm=inp["qk_l2norm"], initial_state=a["initial_state"],
                                    dfinal=a["dfinal"], cu_seqlens=a["cu_seqlens"])
        errs = {}
        for name in ("q", "k", "v", "g", "beta"):
            errs[name] = _check(f"{workload} h={h} d{name}", grads[name][:, :, h:h + 1].double().cpu().numpy(),
                                ref[name])
        errs["A_log"] = _check(f"{workload} h={h} dA_log", grads["A_log"][h:h + 1].double().cpu().numpy(),
                               ref["A_log"])
        errs["dt_bias"] = _check(f"{workload} h={h} ddt_bias", grads["dt_bias"][h:h + 1].double().cpu().numpy(),
                                 ref["dt_bias"])
        if dfin is not None:
            errs["initial_state"] = _check(f"{workload} h={h} dinit",
                                           grads["initial_state"][:, h:h + 1].double().cpu().numpy(),
                                           ref["initial_state"])
        tl.record_grad_margin(f"{workload} full h={h}", errs)


def test_backward_is_deterministic():
    """Two calls on the same inputs give the same bits for every gradient
    (dA_log and dt_bias included: per-chunk parts summed in slot order)."""
    inp = make_inputs(WORKLOADS["packed_varlen"], lengths=[130, 0, 77, 64, 1], H=4, seed=240)
    gen = torch.Generator().manual_seed(241)
    dout = (torch.randn(inp["v"].shape, generator=gen) * 0.5).to(torch.bfloat16).cuda()
    dfin = (torch.randn((inp["N"], 4, 128, 128), generator=gen) * 0.1).cuda()
    d = tl.to_device(inp)

    def call():
        g = K.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], dout, d["A_log"], d["dt_bias"],
                      inp["lower_bound"], d["initial_state"], dfin, d["cu_seqlens"], qk_l2norm=True, gate="safe")
        torch.cuda.synchronize()
        return g

    a, b = call(), call()
    for name, x in a.items():
        if x is not None:
            assert torch.equal(x, b[name]), name
