"""CUDA graph capture of kda_fwd and kda_bwd.

A call captured into a CUDA graph replays to the same bits as the call run
eagerly: for one-pass shapes (short, and two sequences of 256 chunks), a
packed (cu_seqlens) shape with its chunk-index scan, and a shape whose state
stage is split into sequence segments.  The tensor maps of the intra-chunk
stage are kernel parameters, so they are captured by value with the launch.
"""
import pytest
import torch

from kimi_delta_attention_05_gb300 import kda_fwd
from kimi_delta_attention_05_gb300.workloads import WORKLOADS, make_inputs
from tests import kda_testlib as tl

pytestmark = pytest.mark.gpu

CASES = [
    ("one pass", "long_context", dict(T=1000, H=4, seed=90)),
    ("packed", "packed_varlen", dict(lengths=[70, 1, 300, 64], H=2, seed=91)),
    ("one pass, 256 chunks", "long_context", dict(B=2, T=16384, H=4, seed=92)),
    ("sequence split", "long_context", dict(T=16384, H=2, seed=94)),
]


def _call(inp, d, out, fin):
    lb = inp["lower_bound"] if inp["gate"] == "safe" else None
    return kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], out, d["A_log"],
                   d["dt_bias"], lb, d["initial_state"], fin, d["cu_seqlens"],
                   qk_l2norm=inp["qk_l2norm"], gate=inp["gate"])


@pytest.mark.parametrize("tag,workload,kw", CASES, ids=[c[0] for c in CASES])
def test_captured_call_replays_bit_identical(tag, workload, kw):
    inp = make_inputs(WORKLOADS[workload], **kw)
    inp["final_state"] = "f32"
    d = tl.to_device(inp)
    H = d["q"].shape[2]

    def fresh():
        return (torch.full_like(d["v"], float("nan")),
                torch.full((inp["N"], H, 128, 128), float("nan"), device="cuda"))

    out_e, fin_e = fresh()
    _call(inp, d, out_e, fin_e)  # eager; also makes the library's per-device set-up
    torch.cuda.synchronize()

    out_g, fin_g = fresh()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _call(inp, d, out_g, fin_g)  # warm-up on the capturing stream's kind of stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        _call(inp, d, out_g, fin_g)
    for _ in range(3):
        out_g.fill_(float("nan"))
        fin_g.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_g.view(torch.int16), out_e.view(torch.int16)), tag
        assert torch.equal(fin_g, fin_e), tag


def test_eager_call_while_another_stream_captures():
    """A capture of a call stays open on stream X while an eager call runs on
    stream Y.  Every kernel of a call runs on the caller's stream, so Y's work
    neither joins X's capture nor fails; both results equal the eager
    reference bit for bit."""
    from kimi_delta_attention_05_gb300 import kda as K
    inp = make_inputs(WORKLOADS["long_context"], B=2, T=16384, H=4, seed=93)
    inp["final_state"] = "f32"
    d = tl.to_device(inp)
    H = d["q"].shape[2]

    def buffers():
        out = torch.full_like(d["v"], float("nan"))
        fin = torch.full((inp["N"], H, 128, 128), float("nan"), device="cuda")
        args = K.make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], out,
                           d["A_log"], d["dt_bias"], None, None, fin, None, inp["qk_l2norm"],
                           inp["gate"])
        ws = torch.empty(K.workspace_bytes(args), dtype=torch.uint8, device="cuda")
        return out, fin, args, ws

    lib = K.load_library()
    import ctypes
    out_r, fin_r, args_r, ws_r = buffers()
    assert lib.kda_fwd_launches(ctypes.byref(args_r)) == 2  # one pass
    K.kda_fwd_args_call(args_r, ws_r, torch.cuda.current_stream())
    sx, sy = torch.cuda.Stream(), torch.cuda.Stream()
    out_x, fin_x, args_x, ws_x = buffers()
    out_y, fin_y, args_y, ws_y = buffers()
    torch.cuda.synchronize()
    K.kda_fwd_args_call(args_x, ws_x, sx)  # per-stream set-up outside the capture
    K.kda_fwd_args_call(args_y, ws_y, sy)
    torch.cuda.synchronize()
    for t in (out_x, fin_x, out_y, fin_y):
        t.fill_(float("nan"))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=sx, capture_error_mode="relaxed"):
        K.kda_fwd_args_call(args_x, ws_x, sx)
        K.kda_fwd_args_call(args_y, ws_y, sy)  # eager, on another stream, capture still open
    torch.cuda.synchronize()
    assert torch.equal(out_y.view(torch.int16), out_r.view(torch.int16))
    assert torch.equal(fin_y, fin_r)
    assert torch.isnan(out_x.float()).all()  # captured, not run yet
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_x.view(torch.int16), out_r.view(torch.int16))
    assert torch.equal(fin_x, fin_r)


BWD_CASES = [
    ("dense", "long_context", dict(T=1000, H=4, seed=96)),
    ("packed", "packed_varlen", dict(lengths=[70, 1, 0, 300, 64], H=2, seed=97)),
]


@pytest.mark.parametrize("tag,workload,kw", BWD_CASES, ids=[c[0] for c in BWD_CASES])
def test_captured_backward_replays_bit_identical(tag, workload, kw):
    """kda_bwd captured into a CUDA graph (every launch and memset on the
    caller's stream, workspace and gradients preallocated) replays to the bits
    of the eager call."""
    from kimi_delta_attention_05_gb300 import kda as K
    inp = make_inputs(WORKLOADS[workload], **kw)
    d = tl.to_device(inp)
    H = d["q"].shape[2]
    gen = torch.Generator().manual_seed(kw["seed"] + 100)
    dout = (torch.randn(d["v"].shape, generator=gen) * 0.5).to(torch.bfloat16).cuda()
    dfin = (torch.randn((inp["N"], H, 128, 128), generator=gen) * 0.1).cuda()
    lb = inp["lower_bound"] if inp["gate"] == "safe" else None
    a, grads = K.make_bwd_args(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], dout, d["A_log"],
                               d["dt_bias"], lb, d["initial_state"], dfin, d["cu_seqlens"],
                               qk_l2norm=inp["qk_l2norm"], gate=inp["gate"])
    ws = torch.empty(max(K.bwd_workspace_bytes(a), 256), dtype=torch.uint8, device="cuda")
    K.kda_bwd_args_call(a, ws, torch.cuda.current_stream())  # eager reference
    torch.cuda.synchronize()
    ref = {n: t.clone() for n, t in grads.items() if t is not None}
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        K.kda_bwd_args_call(a, ws, side)  # warm-up on a non-default stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        K.kda_bwd_args_call(a, ws, torch.cuda.current_stream())
    for _ in range(2):
        for t in ref:
            grads[t].fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for n, t in ref.items():
            assert torch.equal(grads[n], t), (tag, n)
