"""Failure path on the GPU without a fault: a bounded wait that nothing
satisfies runs out, the kernel records KDA_ERR_DEVICE_TIMEOUT in the status
word of its stream and returns, the host reads it, and the context stays
usable (a normal forward call afterwards is correct).  Status words are per
stream: a call on another stream, in flight at the same time, reads only its
own (clean) word, and reading one stream's word clears nothing else."""
import ctypes

import pytest
import torch

from kimi_delta_attention_05_gb300 import kda as K
from kimi_delta_attention_05_gb300.workloads import WORKLOADS, make_inputs
from tests import kda_testlib as tl

pytestmark = pytest.mark.gpu

KDA_ERR_DEVICE_TIMEOUT = 13


def test_wait_runs_out_sets_status_and_context_survives():
    lib = K.load_library()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    K.get_status(stream)  # start clean
    assert lib.kda_selftest_wait_timeout(1 << 20, ctypes.c_void_p(stream.cuda_stream)) == 0
    torch.cuda.synchronize()
    assert K.get_status(stream) == KDA_ERR_DEVICE_TIMEOUT
    assert K.get_status(stream) == 0  # cleared by the read above
    inp = make_inputs(WORKLOADS["dense_batch"], B=1, T=130, H=2, seed=51)
    o, f = tl.run_gpu(inp)
    ro, rf = tl.run_oracle(inp)
    tl.check_out(o, ro, "after a timed-out wait")
    tl.check_state(f, rf, "after a timed-out wait")
    assert K.get_status(stream) == 0  # the real kernels met every wait


def test_two_streams_each_read_only_their_own_status():
    """Stream A: a wait that runs out (about 2^24 cycles, ~8 ms) with a forward
    call queued behind it; stream B: a forward call issued while A's wait is
    still running.  A reads the timeout, B reads 0, and both results are
    correct.  Reading B's word leaves A's set, and vice versa."""
    lib = K.load_library()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    K.get_status(sa)
    K.get_status(sb)
    inp_a = make_inputs(WORKLOADS["dense_batch"], B=1, T=200, H=2, seed=52)
    inp_b = make_inputs(WORKLOADS["packed_varlen"], lengths=[70, 1, 130], H=2, seed=53)
    assert lib.kda_selftest_wait_timeout(1 << 24, ctypes.c_void_p(sa.cuda_stream)) == 0
    o_b, f_b = tl.run_gpu(inp_b, stream=sb)  # synchronises the device when done
    assert K.get_status(sb) == 0
    o_a, f_a = tl.run_gpu(inp_a, stream=sa)
    assert K.get_status(sa) == KDA_ERR_DEVICE_TIMEOUT
    assert K.get_status(sa) == 0 and K.get_status(sb) == 0
    for inp, o, f, tag in ((inp_a, o_a, f_a, "stream A"), (inp_b, o_b, f_b, "stream B")):
        ro, rf = tl.run_oracle(inp)
        tl.check_out(o, ro, tag)
        tl.check_state(f, rf, tag)
