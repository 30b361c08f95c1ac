"""Failure path on the GPU without a fault: a bounded wait that nothing
satisfies runs out, the kernel sets the device status word and returns, the
host reads KDA_ERR_DEVICE_TIMEOUT, and the context stays usable (a normal
forward call afterwards is correct)."""
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
    lib.kda_get_status(1)  # start clean
    stream = torch.cuda.current_stream()
    assert lib.kda_selftest_wait_timeout(1 << 20, ctypes.c_void_p(stream.cuda_stream)) == 0
    torch.cuda.synchronize()
    assert lib.kda_get_status(1) == KDA_ERR_DEVICE_TIMEOUT
    assert lib.kda_get_status(0) == 0  # cleared by the read above
    inp = make_inputs(WORKLOADS["dense_batch"], B=1, T=130, H=2, seed=51)
    o, f = tl.run_gpu(inp)
    ro, rf = tl.run_oracle(inp)
    tl.check_out(o, ro, "after a timed-out wait")
    tl.check_state(f, rf, "after a timed-out wait")
    assert lib.kda_get_status(0) == 0  # the real kernels met every wait
