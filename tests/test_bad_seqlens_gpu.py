"""Inconsistent cu_seqlens values are caught on the device (KDA_ERR_BAD_SEQLENS).

The values of cu_seqlens are never read on the host by kda_fwd; the kernels
check 0 = cu[0] <= ... <= cu[N] = T.  kda_fwd then processes no sequence
(output untouched, final state = initial state); kda_fwd_recurrent skips the
sequences whose bounds leave [0, T] or decrease; kda_bwd processes no chunk
(zero gradients, dinitial = dfinal).

Every case here is built so that even a broken check could not touch memory
outside the allocations: all cu values are >= 0, token tensors are allocated
for the largest value, and the workspace is four times what is declared.
"""
import ctypes

import numpy as np
import pytest
import torch

from kimi_delta_attention_05_gb300 import kda as K
from kimi_delta_attention_05_gb300.workloads import WORKLOADS, make_inputs
from tests import kda_testlib as tl

pytestmark = pytest.mark.gpu

BAD_SEQLENS = 14


def _call(cu_vals, T_declared, recurrent=False, H=2, seed=80):
    """Run one call with the given cu values; returns (out, final, init, status)."""
    lib = K.load_library()
    rows = max(max(cu_vals), T_declared)
    inp = make_inputs(WORKLOADS["packed_varlen"], lengths=[rows], H=H, seed=seed)
    N = len(cu_vals) - 1
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    init = torch.randn((N, H, 128, 128), generator=torch.Generator().manual_seed(seed + 1)).cuda()
    final = torch.full_like(init, float("nan"))
    out = torch.full_like(d["v"], float("nan"))
    cu = torch.tensor(cu_vals, dtype=torch.int64, device="cuda")
    a = K.make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], out, d["A_log"],
                    d["dt_bias"], inp["lower_bound"], init, final, cu, qk_l2norm=True, gate="safe")
    a.T = T_declared
    stream = torch.cuda.current_stream()
    assert K.get_status(stream) >= 0  # clear
    if recurrent:
        rc = lib.kda_fwd_recurrent(ctypes.byref(a), ctypes.c_void_p(stream.cuda_stream))
    else:
        need = int(lib.kda_fwd_workspace_bytes(ctypes.byref(a)))
        ws = torch.empty(4 * need + (1 << 20), dtype=torch.uint8, device="cuda")
        rc = lib.kda_fwd(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), need,
                         ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    status = K.get_status(stream)
    return out, final, init, status


@pytest.mark.parametrize("cu_vals,T", [
    ([0, 300, 100, 400], 400),   # decreasing: sequences would overlap
    ([0, 100, 264], 200),        # cu[N] > T
    ([10, 100, 200], 200),       # cu[0] != 0
    ([0, 150, 120], 120),        # decreasing at the end, cu[N] == T
])
def test_chunked_path_skips_every_sequence(cu_vals, T):
    out, final, init, status = _call(cu_vals, T)
    assert status == BAD_SEQLENS
    assert torch.isnan(out.float()).all()        # no output row written
    assert torch.equal(final, init)              # final state = initial state


def test_recurrent_path_skips_only_bad_sequences():
    cu_vals = [0, 40, 10, 60]  # sequence 1 decreases; sequences 0 and 2 are in range
    out, final, init, status = _call(cu_vals, 60, recurrent=True)
    assert status == BAD_SEQLENS
    assert torch.equal(final[1], init[1])
    assert not torch.equal(final[0], init[0]) and not torch.equal(final[2], init[2])


def test_valid_call_after_a_bad_one_is_clean():
    _call([0, 300, 100, 400], 400)
    inp = make_inputs(WORKLOADS["packed_varlen"], lengths=[130, 0, 70], H=2, seed=81)
    o, f = tl.run_gpu(inp)
    assert K.get_status() == 0
    ro, rf = tl.run_oracle(inp)
    tl.check_out(o, ro, "after bad call")
    tl.check_state(f, rf, "after bad call")


@pytest.mark.parametrize("cu_vals,T", [
    ([0, 300, 100, 400], 400),   # decreasing: sequences would overlap
    ([0, 100, 264], 200),        # cu[N] > T
    ([0, 150, 120], 120),        # decreasing at the end, cu[N] == T
])
def test_backward_skips_every_sequence(cu_vals, T):
    """kda_bwd with inconsistent cu_seqlens processes no chunk: zero token
    gradients, zero dA_log and dt_bias sums, dinitial = dfinal, and the
    stream's status word reads KDA_ERR_BAD_SEQLENS."""
    lib = K.load_library()
    H, seed = 2, 90
    rows = max(max(cu_vals), T)
    inp = make_inputs(WORKLOADS["packed_varlen"], lengths=[rows], H=H, seed=seed)
    N = len(cu_vals) - 1
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    gen = torch.Generator().manual_seed(seed + 1)
    init = torch.randn((N, H, 128, 128), generator=gen).cuda()
    dfin = torch.randn((N, H, 128, 128), generator=gen).cuda()
    dout = torch.randn(d["v"].shape, generator=gen).to(torch.bfloat16).cuda()
    cu = torch.tensor(cu_vals, dtype=torch.int64, device="cuda")
    a, grads = K.make_bwd_args(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], dout, d["A_log"],
                               d["dt_bias"], inp["lower_bound"], init, dfin, cu, qk_l2norm=True, gate="safe")
    a.fwd.T = T
    for t in grads.values():
        if t is not None:
            t.fill_(float("nan"))
    stream = torch.cuda.current_stream()
    assert K.get_status(stream) >= 0  # clear
    need = int(lib.kda_bwd_workspace_bytes(ctypes.byref(a)))
    ws = torch.empty(4 * need + (1 << 20), dtype=torch.uint8, device="cuda")
    rc = lib.kda_bwd(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), need, ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert K.get_status(stream) == BAD_SEQLENS
    for name in ("q", "k", "v", "g", "beta"):
        assert torch.count_nonzero(grads[name][:, :T]) == 0, name
    assert torch.count_nonzero(grads["A_log"]) == 0 and torch.count_nonzero(grads["dt_bias"]) == 0
    assert torch.equal(grads["initial_state"], dfin)
