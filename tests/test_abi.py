"""C-ABI checks that need no GPU: the library loads, exports every function
declared in include/kda.h, and rejects each invalid argument set with its
error code before anything is launched (no call below has a valid argument
set, so no kernel can start)."""
import ctypes
import os
import re
import subprocess

import pytest

from kimi_delta_attention_05_gb300 import kda as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x7F0000000000  # 256-byte aligned, never dereferenced


def declared_functions():
    names = []
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if hdr.endswith(".h"):
            text = open(os.path.join(ROOT, "include", hdr)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(kda_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_declared_symbols():
    lib = K.load_library()
    names = declared_functions()
    assert {"kda_fwd", "kda_fwd_workspace_bytes", "kda_error_string", "kda_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", K.library_path()], capture_output=True,
                         text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}\b", out), f"{n} missing from the dynamic symbol table"


def _valid_args(**over):
    a = K.kda_fwd_args()
    for f in ("q", "k", "v", "g", "beta", "out"):
        setattr(a, f, FAKE)
    a.scale = 0.088
    a.A_log = FAKE
    a.dt_bias = FAKE
    a.lower_bound = -5.0
    a.state_dtype = K.KDA_DTYPE_F32
    a.B, a.T, a.H, a.N, a.K, a.V = 2, 100, 4, 2, 128, 128
    a.flags = K.KDA_GATE_SAFE | K.KDA_QK_L2NORM
    for k_, v in over.items():
        setattr(a, k_, v)
    return a


def _call(a, ws=None, nbytes=0):
    lib = K.load_library()
    return lib.kda_fwd(ctypes.byref(a), ws, nbytes, None)


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1), (dict(out=None), 1), (dict(beta=None), 1),
    (dict(K=64), 2), (dict(V=256), 2),
    (dict(T=-1), 3), (dict(N=3), 3), (dict(H=70000), 3),
    (dict(flags=0), 4), (dict(flags=3), 4), (dict(flags=1 | 0x100), 4), (dict(flags=1 | 0x40), 4),
    (dict(flags=K.KDA_GATE_LOGSPACE | K.KDA_GATE_SAFE), 4),
    (dict(flags=K.KDA_GATE_LOGSPACE | K.KDA_GATE_UNSAFE), 4),
    (dict(lower_bound=0.0), 5), (dict(lower_bound=-5.5), 5), (dict(lower_bound=float("nan")), 5),
    (dict(flags=K.KDA_GATE_UNSAFE, A_log=None), 6),
    (dict(initial_state=FAKE, state_dtype=7), 7),
    (dict(cu_seqlens=FAKE, B=2), 8),
    (dict(q=FAKE + 2), 9), (dict(initial_state=FAKE + 8), 9), (dict(cu_seqlens=FAKE + 4, B=1), 9),
])
def test_invalid_arguments_rejected(over, code):
    a = _valid_args(**over)
    assert _call(a, FAKE, 1 << 40) == code
    assert K.load_library().kda_fwd_workspace_bytes(ctypes.byref(a)) == 0


def test_logspace_gate_and_beta_prob_accepted():
    """The caller-gated mode needs no A_log and ignores lower_bound; beta given
    as beta itself combines with any gate form."""
    lib = K.load_library()
    for flags in (K.KDA_GATE_LOGSPACE, K.KDA_GATE_LOGSPACE | K.KDA_BETA_PROB,
                  K.KDA_GATE_UNSAFE | K.KDA_BETA_PROB | K.KDA_QK_L2NORM,
                  K.KDA_GATE_LOGSPACE | K.KDA_G_FP32, K.KDA_GATE_UNSAFE | K.KDA_G_FP32):
        a = _valid_args(flags=flags, A_log=None if flags & K.KDA_GATE_LOGSPACE else FAKE,
                        lower_bound=0.0)
        assert lib.kda_fwd_workspace_bytes(ctypes.byref(a)) > 0


def test_wait_selftest_rejects_bad_limits_before_launch():
    lib = K.load_library()
    assert lib.kda_selftest_wait_timeout(0, None) == 3
    assert lib.kda_selftest_wait_timeout(1 << 40, None) == 3


def test_workspace_checked_before_launch():
    a = _valid_args()
    need = K.load_library().kda_fwd_workspace_bytes(ctypes.byref(a))
    assert need == 2 * 2 * 4 * 74240  # B * ceil(T/64) * H slots of 74240 bytes
    assert _call(a, None, need) == 10
    assert _call(a, FAKE, need - 1) == 10
    assert _call(a, FAKE + 16, need) == 10  # not 256-byte aligned


def test_workspace_varlen_size():
    a = _valid_args(B=1, T=1000, N=5, cu_seqlens=FAKE)
    need = K.load_library().kda_fwd_workspace_bytes(ctypes.byref(a))
    assert need == 256 + (16 + 5) * 4 * 74240


def test_launch_count():
    """kda_fwd_launches: the chunk and state kernels (2), plus the chunk-index
    scan with cu_seqlens (3), only the state kernel with no tokens (1), none for
    argument sets kda_fwd rejects (0).  These sequences are far too short for
    the token-range split, so the counts hold with or without a device."""
    lib = K.load_library()
    assert lib.kda_fwd_launches(ctypes.byref(_valid_args())) == 2
    assert lib.kda_fwd_launches(ctypes.byref(_valid_args(B=1, T=1000, N=5, cu_seqlens=FAKE))) == 3
    assert lib.kda_fwd_launches(ctypes.byref(_valid_args(T=0))) == 1
    assert lib.kda_fwd_launches(ctypes.byref(_valid_args(K=64))) == 0
    assert lib.kda_fwd_launches(ctypes.byref(_valid_args(flags=0))) == 0


def test_error_strings():
    lib = K.load_library()
    for c in range(12):
        assert lib.kda_error_string(c)
    assert b"unknown" in lib.kda_error_string(99)
    assert lib.kda_version() >= 100


# ---- kda_fwd_host: argument checks and device-buffer size (no GPU touched) ----

def _host_call(a, buf=None, nbytes=0):
    return K.load_library().kda_fwd_host(ctypes.byref(a), buf, nbytes, None)


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1), (dict(K=64), 2), (dict(N=3), 3), (dict(flags=0), 4),
    (dict(lower_bound=0.0), 5), (dict(flags=K.KDA_GATE_UNSAFE, A_log=None), 6),
    (dict(initial_state=FAKE, state_dtype=7), 7), (dict(cu_seqlens=FAKE, B=2), 8),
    (dict(q=FAKE + 2), 9),
])
def test_host_entry_rejects_like_kda_fwd(over, code):
    a = _valid_args(**over)
    assert _host_call(a, FAKE, 1 << 40) == code
    assert K.load_library().kda_fwd_host_device_bytes(ctypes.byref(a)) == 0


def test_host_device_bytes_dense_single_piece():
    """B=2, T=100, H=4, no states: device copies of q, k, v, g, out, beta,
    A_log, dt_bias and one piece's workspace, each region 256-byte aligned."""
    a = _valid_args()
    need = K.load_library().kda_fwd_host_device_bytes(ctypes.byref(a))
    rows = 2 * 100
    qlike = rows * 4 * 256
    assert need == 5 * qlike + 1792 + 256 + 2048 + 2 * 2 * 4 * 74240
    assert _host_call(a, None, need) == 10
    assert _host_call(a, FAKE, need - 1) == 10
    assert _host_call(a, FAKE + 16, need) == 10


def test_host_device_bytes_dense_pieces_carry_state():
    """Past 32 MiB of inputs a dense call is cut into token-range pieces: the
    workspace is one piece's and an fp32 state carry appears."""
    import numpy as np
    a = _valid_args(B=1, N=1, T=16384, H=4)
    need = K.load_library().kda_fwd_host_device_bytes(ctypes.byref(a))
    qlike = 16384 * 4 * 256
    beta = 16384 * 4 * 2
    carry = 1 * 4 * 128 * 128 * 4
    ws = 1 * (5504 // 64) * 4 * 74240  # three pieces of at most 5504 tokens
    assert need == 5 * qlike + beta + 256 + 2048 + carry + ws
    assert np.int64(need) > 0


def test_host_cu_seqlens_checked_on_host():
    import numpy as np
    lib = K.load_library()
    for bad in ([0, 10, 5, 100], [0, 10, 50, 99], [1, 10, 50, 100]):
        cu = np.array(bad, dtype=np.int64)
        a = _valid_args(B=1, T=100, N=3, cu_seqlens=cu.ctypes.data)
        assert _host_call(a, FAKE, 1 << 40) == 3
        assert lib.kda_fwd_host_device_bytes(ctypes.byref(a)) == 0
    cu = np.array([0, 10, 10, 100], dtype=np.int64)
    a = _valid_args(B=1, T=100, N=3, cu_seqlens=cu.ctypes.data)
    need = lib.kda_fwd_host_device_bytes(ctypes.byref(a))
    qlike = 100 * 4 * 256
    ws = 256 + (2 + 3) * 4 * 74240  # one group of all three sequences
    # q, k, v, g, out; beta; A_log; dt_bias; cu; the group's cu from 0; workspace
    assert need == 5 * qlike + 1024 + 256 + 2048 + 256 + 256 + ws


def test_no_tokens_allows_null_token_tensors():
    """B * T == 0: the token tensors may be NULL (empty torch tensors have no
    storage); with tokens they may not."""
    lib = K.load_library()
    empty = dict(q=None, k=None, v=None, g=None, beta=None, out=None, T=0)
    a = _valid_args(**empty)
    assert lib.kda_fwd_host_device_bytes(ctypes.byref(a)) == 256 + 2048  # A_log, dt_bias
    assert _host_call(a, None, 0) == 10  # past the argument checks: wants its buffer
    assert _host_call(_valid_args(q=None), None, 0) == 1


def test_fp32_g_doubles_the_g_region_of_the_host_buffer():
    lib = K.load_library()
    a16 = _valid_args()
    a32 = _valid_args(flags=K.KDA_GATE_SAFE | K.KDA_QK_L2NORM | K.KDA_G_FP32)
    d16 = lib.kda_fwd_host_device_bytes(ctypes.byref(a16))
    d32 = lib.kda_fwd_host_device_bytes(ctypes.byref(a32))
    assert d32 - d16 == 2 * 100 * 4 * 256  # B * T * H rows of 256 more bytes
