"""GB300-native Kimi Delta Attention (KDA): chunked forward pass and its backward pass.

The compute path is ``libkda.so`` (CUDA, sm_103a; C ABI in include/kda.h);
this package holds its build script, a thin ctypes binding and the seeded
workload generator.
"""
from .kda import (kda_bwd, kda_fwd, kda_fwd_host, kda_fwd_recurrent, get_status, load_library,  # noqa: F401
                  KdaError, workspace_bytes)
from . import workloads  # noqa: F401

__version__ = "0.1.0"
