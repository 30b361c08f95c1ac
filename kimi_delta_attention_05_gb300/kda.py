"""Thin Python binding of libkda (include/kda.h).

Argument marshalling only: every step of the forward pass runs in the CUDA
library.  PyTorch supplies device memory and the stream.  If the library is
missing this raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

KDA_GATE_SAFE = 0x1
KDA_GATE_UNSAFE = 0x2
KDA_QK_L2NORM = 0x4
KDA_GATE_LOGSPACE = 0x8
KDA_BETA_PROB = 0x10
KDA_G_FP32 = 0x20
KDA_DTYPE_F32 = 0
KDA_DTYPE_BF16 = 1
HEAD_DIM = 128


class KdaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"kda_fwd failed with status {code}: {msg}")
        self.code = code


class kda_fwd_args(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("scale", ctypes.c_float),
        ("out", ctypes.c_void_p),
        ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("lower_bound", ctypes.c_float),
        ("initial_state", ctypes.c_void_p), ("final_state", ctypes.c_void_p),
        ("state_dtype", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p),
        ("B", ctypes.c_int64), ("T", ctypes.c_int64), ("H", ctypes.c_int64), ("N", ctypes.c_int64),
        ("K", ctypes.c_int64), ("V", ctypes.c_int64),
        ("flags", ctypes.c_uint32),
    ]


class kda_bwd_args(ctypes.Structure):
    _fields_ = [
        ("fwd", kda_fwd_args),
        ("dout", ctypes.c_void_p), ("dfinal_state", ctypes.c_void_p),
        ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("dg", ctypes.c_void_p), ("dbeta", ctypes.c_void_p), ("dA_log", ctypes.c_void_p),
        ("ddt_bias", ctypes.c_void_p), ("dinitial_state", ctypes.c_void_p),
    ]


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True):
    """Load libkda.so (building it first if asked and needed)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libkda.so not found at {path}; run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        lib.kda_fwd.restype = ctypes.c_int
        lib.kda_fwd.argtypes = [ctypes.POINTER(kda_fwd_args), P, ctypes.c_size_t, P]
        lib.kda_fwd_workspace_bytes.restype = ctypes.c_size_t
        lib.kda_fwd_workspace_bytes.argtypes = [ctypes.POINTER(kda_fwd_args)]
        lib.kda_error_string.restype = ctypes.c_char_p
        lib.kda_error_string.argtypes = [ctypes.c_int]
        lib.kda_version.restype = ctypes.c_int
        lib.kda_fwd_profiled.restype = ctypes.c_int
        lib.kda_fwd_profiled.argtypes = [ctypes.POINTER(kda_fwd_args), P, ctypes.c_size_t, P,
                                         ctypes.POINTER(ctypes.c_void_p)]
        lib.kda_fwd_launches.restype = ctypes.c_int
        lib.kda_fwd_launches.argtypes = [ctypes.POINTER(kda_fwd_args)]
        lib.kda_get_status.restype = ctypes.c_int
        lib.kda_get_status.argtypes = [P]
        lib.kda_selftest_wait_timeout.restype = ctypes.c_int
        lib.kda_selftest_wait_timeout.argtypes = [ctypes.c_longlong, P]
        lib.kda_fwd_host.restype = ctypes.c_int
        lib.kda_fwd_host.argtypes = [ctypes.POINTER(kda_fwd_args), P, ctypes.c_size_t, P]
        lib.kda_fwd_host_device_bytes.restype = ctypes.c_size_t
        lib.kda_fwd_host_device_bytes.argtypes = [ctypes.POINTER(kda_fwd_args)]
        lib.kda_fwd_recurrent.restype = ctypes.c_int
        lib.kda_fwd_recurrent.argtypes = [ctypes.POINTER(kda_fwd_args), P]
        lib.kda_bwd.restype = ctypes.c_int
        lib.kda_bwd.argtypes = [ctypes.POINTER(kda_bwd_args), P, ctypes.c_size_t, P]
        lib.kda_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.kda_bwd_workspace_bytes.argtypes = [ctypes.POINTER(kda_bwd_args)]
        lib.kda_bwd_profiled.restype = ctypes.c_int
        lib.kda_bwd_profiled.argtypes = [ctypes.POINTER(kda_bwd_args), P, ctypes.c_size_t, P,
                                         ctypes.POINTER(ctypes.c_void_p)]
        _lib = lib
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def make_args(q, k, v, g, beta, scale, out, A_log=None, dt_bias=None, lower_bound=None,
              initial_state=None, final_state=None, cu_seqlens=None, qk_l2norm=False,
              gate=None, beta_prob=False) -> kda_fwd_args:
    """Build the C argument block from tensors (no checks beyond shapes;
    the library validates).  ``gate``: "safe", "unsafe" or "logspace" (g holds
    the log decay); default from ``lower_bound``.  ``beta_prob``: beta holds
    beta itself instead of logits.  A float32 ``g`` sets KDA_G_FP32."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    if gate is None:
        gate = "unsafe" if lower_bound is None else "safe"
    flags = {"safe": KDA_GATE_SAFE, "unsafe": KDA_GATE_UNSAFE, "logspace": KDA_GATE_LOGSPACE}[gate]
    if qk_l2norm:
        flags |= KDA_QK_L2NORM
    if beta_prob:
        flags |= KDA_BETA_PROB
    if g is not None and g.dtype == torch.float32:
        flags |= KDA_G_FP32
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    st = initial_state if initial_state is not None else final_state
    sd = KDA_DTYPE_BF16 if (st is not None and st.dtype == torch.bfloat16) else KDA_DTYPE_F32
    a = kda_fwd_args()
    a.q, a.k, a.v, a.g, a.beta = _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta)
    a.scale = float(scale)
    a.out = _ptr(out)
    a.A_log, a.dt_bias = _ptr(A_log), _ptr(dt_bias)
    a.lower_bound = float(lower_bound if lower_bound is not None else 0.0)
    a.initial_state, a.final_state = _ptr(initial_state), _ptr(final_state)
    a.state_dtype = sd
    a.cu_seqlens = _ptr(cu_seqlens)
    a.B, a.T, a.H, a.N, a.K, a.V = B, T, H, N, K, V
    a.flags = flags
    return a


def get_status(stream=None) -> int:
    """Read and clear the device status word of ``stream`` (a torch stream;
    default: the current stream): 0, KDA_ERR_DEVICE_TIMEOUT (13) or
    KDA_ERR_BAD_SEQLENS (14) for the calls enqueued on it; -1 if it cannot be
    read.  Synchronises the stream."""
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(load_library().kda_get_status(ctypes.c_void_p(s.cuda_stream)))


def workspace_bytes(args: kda_fwd_args) -> int:
    return int(load_library().kda_fwd_workspace_bytes(ctypes.byref(args)))


def kda_fwd(q, k, v, g, beta, scale, out=None, A_log=None, dt_bias=None, lower_bound=None,
            initial_state=None, final_state=None, cu_seqlens=None, *, qk_l2norm=False,
            gate=None, beta_prob=False, workspace=None, stream=None):
    """KDA chunked forward on device tensors; returns ``out``.

    Mirrors the flashkda.fwd argument list: q, k, g [B,T,H,128] bf16, v
    [B,T,H,128] bf16, beta [B,T,H] bf16 logits, out [B,T,H,128] bf16
    (allocated here if None), A_log [H] fp32, dt_bias [H,128] fp32,
    lower_bound (None -> unsafe softplus gate), initial/final state
    [N,H,128,128] fp32 or bf16, cu_seqlens [N+1] int64.  ``workspace`` is an
    optional pre-allocated uint8 device tensor; ``stream`` a torch stream.
    """
    lib = load_library()
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    # buffers made here are allocated on the stream that uses them, so the
    # caching allocator does not hand them out again while that stream runs
    with torch.cuda.stream(s):
        if out is None:
            out = torch.empty_like(v)
        a = make_args(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                      final_state, cu_seqlens, qk_l2norm, gate, beta_prob)
        need = int(lib.kda_fwd_workspace_bytes(ctypes.byref(a)))
        if workspace is None or workspace.numel() < need:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    rc = lib.kda_fwd(ctypes.byref(a), ctypes.c_void_p(workspace.data_ptr()), need,
                     ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise KdaError(rc, lib.kda_error_string(rc).decode())
    return out


def kda_fwd_recurrent(q, k, v, g, beta, scale, out=None, A_log=None, dt_bias=None,
                      lower_bound=None, initial_state=None, final_state=None, cu_seqlens=None, *,
                      qk_l2norm=False, gate=None, beta_prob=False, stream=None):
    """Token-by-token forward (decoding path, no workspace); same arguments as
    :func:`kda_fwd`.  ``final_state`` may be ``initial_state`` itself."""
    lib = load_library()
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    if out is None:
        with torch.cuda.stream(s):
            out = torch.empty_like(v)
    a = make_args(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                  final_state, cu_seqlens, qk_l2norm, gate, beta_prob)
    rc = lib.kda_fwd_recurrent(ctypes.byref(a), ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise KdaError(rc, lib.kda_error_string(rc).decode())
    return out


def kda_fwd_args_call(args: kda_fwd_args, workspace, stream, events=None) -> None:
    """Call the library on a prepared argument block (used by the benchmark to
    keep Python marshalling out of the timed loop).  ``events``: optional
    three raw cudaEvent_t handles (ints) for kda_fwd_profiled."""
    lib = load_library()
    need = int(lib.kda_fwd_workspace_bytes(ctypes.byref(args)))
    wptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else None
    if events is None:
        rc = lib.kda_fwd(ctypes.byref(args), wptr, need, ctypes.c_void_p(stream.cuda_stream))
    else:
        arr = (ctypes.c_void_p * 3)(*[ctypes.c_void_p(e) if e else None for e in events])
        rc = lib.kda_fwd_profiled(ctypes.byref(args), wptr, need,
                                  ctypes.c_void_p(stream.cuda_stream), arr)
    if rc != 0:
        raise KdaError(rc, lib.kda_error_string(rc).decode())


def kda_fwd_host(q, k, v, g, beta, scale, out=None, A_log=None, dt_bias=None, lower_bound=None,
                 initial_state=None, final_state=None, cu_seqlens=None, *, qk_l2norm=False,
                 gate=None, beta_prob=False, device_buffer=None, stream=None, device=None):
    """End-to-end forward on HOST (CPU) tensors through ``kda_fwd_host``: the
    library copies the inputs in, runs the path and copies ``out`` (and
    ``final_state``) back, pipelining the copies with the kernels.  Tensors
    should be pinned (``.pin_memory()``) for the copies to overlap.  Same
    arguments as :func:`kda_fwd`, all on the CPU; ``device_buffer`` is an
    optional uint8 CUDA tensor of at least :func:`host_device_bytes` bytes.
    Asynchronous on ``stream``: synchronise it before reading the results.
    Returns ``out``."""
    lib = load_library()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if out is None:
        out = torch.empty(v.shape, dtype=v.dtype, pin_memory=v.is_pinned())
    a = make_args(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                  final_state, cu_seqlens, qk_l2norm, gate, beta_prob)
    need = int(lib.kda_fwd_host_device_bytes(ctypes.byref(a)))
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    if device_buffer is None or device_buffer.numel() < need:
        with torch.cuda.stream(s):  # allocated on the stream that uses it
            device_buffer = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    rc = lib.kda_fwd_host(ctypes.byref(a), ctypes.c_void_p(device_buffer.data_ptr()), need,
                          ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise KdaError(rc, lib.kda_error_string(rc).decode())
    return out


def host_device_bytes(args: kda_fwd_args) -> int:
    """Device buffer bytes kda_fwd_host needs for an argument block of host
    pointers (0 for an invalid one)."""
    return int(load_library().kda_fwd_host_device_bytes(ctypes.byref(args)))


def kda_fwd_host_args_call(args: kda_fwd_args, device_buffer, stream) -> None:
    """kda_fwd_host on a prepared argument block of host pointers (keeps
    Python marshalling out of a timed loop)."""
    lib = load_library()
    need = int(lib.kda_fwd_host_device_bytes(ctypes.byref(args)))
    rc = lib.kda_fwd_host(ctypes.byref(args), ctypes.c_void_p(device_buffer.data_ptr()), need,
                          ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise KdaError(rc, lib.kda_error_string(rc).decode())


def make_bwd_args(q, k, v, g, beta, scale, dout, A_log=None, dt_bias=None, lower_bound=None,
                  initial_state=None, dfinal_state=None, cu_seqlens=None, *, qk_l2norm=False,
                  gate=None, beta_prob=False):
    """The argument block of ``kda_bwd`` and freshly allocated fp32 gradient
    tensors (same conventions as :func:`kda_bwd`): returns (args, grads)."""
    gate_name = gate if gate is not None else ("unsafe" if lower_bound is None else "safe")
    f32 = dict(dtype=torch.float32, device=q.device)
    grads = {"q": torch.empty(q.shape, **f32), "k": torch.empty(k.shape, **f32),
             "v": torch.empty(v.shape, **f32), "g": torch.empty(g.shape, **f32),
             "beta": torch.empty(beta.shape, **f32)}
    gate_params = gate_name != "logspace"
    grads["A_log"] = torch.empty(A_log.shape, **f32) if (A_log is not None and gate_params) else None
    grads["dt_bias"] = torch.empty(dt_bias.shape, **f32) if (dt_bias is not None and gate_params) else None
    grads["initial_state"] = torch.empty(initial_state.shape, **f32) if initial_state is not None else None
    a = kda_bwd_args()
    a.fwd = make_args(q, k, v, g, beta, scale, None, A_log, dt_bias, lower_bound, initial_state,
                      None, cu_seqlens, qk_l2norm, gate, beta_prob)
    a.dout = _ptr(dout)
    a.dfinal_state = _ptr(dfinal_state)
    a.dq, a.dk, a.dv, a.dg = _ptr(grads["q"]), _ptr(grads["k"]), _ptr(grads["v"]), _ptr(grads["g"])
    a.dbeta = _ptr(grads["beta"])
    a.dA_log, a.ddt_bias = _ptr(grads["A_log"]), _ptr(grads["dt_bias"])
    a.dinitial_state = _ptr(grads["initial_state"])
    return a, grads


def bwd_workspace_bytes(args: kda_bwd_args) -> int:
    return int(load_library().kda_bwd_workspace_bytes(ctypes.byref(args)))


def kda_bwd_args_call(args: kda_bwd_args, workspace, stream, events=None) -> None:
    """Call ``kda_bwd`` on a prepared argument block (``events``: optional four
    raw cudaEvent_t handles for ``kda_bwd_profiled``)."""
    lib = load_library()
    need = int(lib.kda_bwd_workspace_bytes(ctypes.byref(args)))
    wptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else None
    if events is None:
        rc = lib.kda_bwd(ctypes.byref(args), wptr, need, ctypes.c_void_p(stream.cuda_stream))
    else:
        arr = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(e) if e else None for e in events])
        rc = lib.kda_bwd_profiled(ctypes.byref(args), wptr, need, ctypes.c_void_p(stream.cuda_stream), arr)
    if rc != 0:
        raise KdaError(rc, lib.kda_error_string(rc).decode())


def kda_bwd(q, k, v, g, beta, scale, dout, A_log=None, dt_bias=None, lower_bound=None,
            initial_state=None, dfinal_state=None, cu_seqlens=None, *, qk_l2norm=False,
            gate=None, beta_prob=False, workspace=None, stream=None):
    """Backward pass through ``kda_bwd``: gradients of <out, dout> +
    <final_state, dfinal_state> for the forward call with these arguments
    (same conventions as :func:`kda_fwd`).  Returns a dict of fp32 device
    tensors: q, k, v, g, beta, A_log (None unless A_log given and the gate is
    not logspace), dt_bias (likewise), initial_state (None unless given)."""
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.stream(s):
        a, grads = make_bwd_args(q, k, v, g, beta, scale, dout, A_log, dt_bias, lower_bound,
                                 initial_state, dfinal_state, cu_seqlens, qk_l2norm=qk_l2norm,
                                 gate=gate, beta_prob=beta_prob)
        need = bwd_workspace_bytes(a)
        if workspace is None or workspace.numel() < need:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    kda_bwd_args_call(a, workspace, s)
    return grads
