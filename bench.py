#!/usr/bin/env python3
"""Benchmark of the KDA chunked forward pass on GB300.

One step = one kda_fwd call over the whole workload (all stages of the path),
inputs resident in HBM.  Prints ONE JSON line (rank 0):

  value      tokens/s over all ranks (tokens = sequence tokens, heads not
             multiplied in), device-timed with CUDA events
  tflops     algorithmic TFLOP/s (132,693 flop per token-head)
  roofline   dominant kernel: its algorithmic bytes / its average duration,
             against the measured HBM copy bandwidth; plus the whole path
  e2e        same metric through the C-ABI host-buffer call (kda_fwd_host) on
             pinned host buffers: host->device inputs and device->host
             outputs inside the timing, pipelined with the kernels
  cpu_baseline  the fp64 oracle on a bounded sample, on the host cores

``--impl reference`` times the oracle itself as the reference arm.
Multi-GPU (torchrun): every rank runs its own copy of the workload (seed +
rank), no collective on the data path ("weak" scaling); only the timing uses a
barrier and a max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from kimi_delta_attention_05_gb300.workloads import WORKLOADS, make_inputs  # noqa: E402

METRIC = "KDA fwd tokens/s, TFLOP/s and % of roofline (bf16 TC/HBM), 1 GB300"
CHUNK, K_DIM = 64, 128
# algorithmic work per token-head (chunk 64, K = V = 128): state products 6KV,
# intra-chunk A and P 2CK, T [V | K gamma] (C+1)(K+V), triangular solve C^2/3
FLOP_PER_TOKEN_HEAD = 6 * K_DIM * K_DIM + 2 * CHUNK * K_DIM + (CHUNK + 1) * 2 * K_DIM + CHUNK ** 2 / 3
# compulsory bytes per token-head: q, k, v, g (bf16 x 128 each) + beta + out
BYTES_IN_PER_TOKEN_HEAD = 4 * 2 * K_DIM + 2
BYTES_OUT_PER_TOKEN_HEAD = 2 * K_DIM
DEFAULT_STEPS = {"tiny": 2000, "dense_batch": 3000, "long_context": 3000, "packed_varlen": 500,
                 "extremes": 1000, "long_sequence": 1000}
KERNEL_SOURCES = {
    "kda_chunk_kernel": ["kda_chunk.cu", "kda_common.cuh", "kda_kernels.cuh", "kda_tc.cuh"],
    "kda_state_kernel": ["kda_state.cu", "kda_common.cuh", "kda_kernels.cuh", "kda_tc.cuh"],
    "kda_recurrent_kernel": ["kda_recurrent.cu", "kda_common.cuh", "kda_kernels.cuh"],
}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="long_context", choices=sorted(WORKLOADS))
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU work of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--path", choices=["chunked", "recurrent", "backward"], default="chunked",
                   help="recurrent: time the token-by-token (decoding) entry point on the "
                        "decode workload instead of the chunked path; backward: time kda_bwd "
                        "(gradients of every input) on the workload")
    return p.parse_args()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def sm_max_mhz():
    """Maximum SM clock: MEASURED_PEAKS.json's record, else the part's 2070 MHz."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if d.get("sm_max_mhz"):
            return float(d["sm_max_mhz"])
    return 2070.0


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "kimi_delta_attention_05_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes (read + write) per launch from the committed ncu summary
    table profiles/traffic.txt, if it was taken on the current source of the
    kernel; else None.  Line format: kernel workload source_hash bytes."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) == 4 and not line.startswith("#") and parts[0] == kernel \
                and parts[1] == workload and parts[2] == kernel_source_hash(kernel):
            return float(parts[3])
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed loop runs."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self, t0=None, t1=None):
        """Median SM clock and active throttle reasons of the samples taken
        between host wall times t0 and t1 (all samples if none fall inside)."""
        import datetime
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 is not None and t0 - 0.06 <= r[0] <= t1 + 0.06]
        use = inside or rows
        sm = [r[1] for r in use]
        mx = use[-1][2] if use else None
        reasons = set()
        for r in use:
            for n, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "samples_in_timed_region": len(inside),
                "sm_mhz_samples": [r[1] for r in use]}


# ---------------------------------------------------------------------------
# workload helpers
# ---------------------------------------------------------------------------

def token_heads(inp):
    q = inp["q"]
    return int(q.shape[0] * q.shape[1] * q.shape[2])


def state_io_bytes(inp):
    H = inp["q"].shape[2]
    b = 0
    if inp["initial_state"] is not None:
        b += inp["initial_state"].numel() * inp["initial_state"].element_size()
    if inp["final_state"] is not None:
        b += inp["N"] * H * K_DIM * K_DIM * (2 if inp["final_state"] == "bf16" else 4)
    return b


def device_call(inp, dev):
    """Device copies of the inputs, the output buffers, the argument block and
    the workspace, for the timed loop."""
    from kimi_delta_attention_05_gb300 import kda as K
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}
    out = torch.empty_like(d["v"])
    fin = None
    if inp["final_state"] is not None:
        dt = torch.bfloat16 if inp["final_state"] == "bf16" else torch.float32
        fin = torch.empty((inp["N"], d["q"].shape[2], K_DIM, K_DIM), dtype=dt, device=dev)
    lb = inp["lower_bound"] if inp["gate"] == "safe" else None
    args = K.make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], out, d["A_log"],
                       d["dt_bias"], lb, d["initial_state"], fin, d["cu_seqlens"],
                       inp["qk_l2norm"], inp["gate"])
    ws = torch.empty(max(K.workspace_bytes(args), 256), dtype=torch.uint8, device=dev)
    return d, out, fin, args, ws


# ---------------------------------------------------------------------------
# multi-rank host logic (also exercised with the gloo backend on CPU by the tests)
# ---------------------------------------------------------------------------

def rank_inputs(w, rank):
    """Every rank runs its own copy of the workload, seeded seed + rank."""
    return make_inputs(w, seed=w.seed + rank)


def max_over_ranks(ms, world, device="cpu"):
    """The timed region's duration is the slowest rank's (all ranks call this)."""
    if world <= 1:
        return float(ms)
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(tokens_per_rank, world, ms_step):
    """tokens/s over all ranks (weak scaling: every rank does the same work)."""
    return tokens_per_rank * world / (ms_step * 1e-3)


class L2Flush:
    """Untimed L2 flush between timed calls: write one buffer larger than the
    129 MB L2, then read another, so that the next call starts with none of its
    own data in L2 and with clean (not dirty) lines to evict."""
    BYTES = 256 << 20

    def __init__(self, dev):
        self.w = torch.empty(self.BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(self.BYTES // 4, dtype=torch.float32, device=dev)
        self.i = 0

    def __call__(self):
        self.i += 1
        self.w.fill_(float(self.i))
        return self.r.sum()


def run_ours(a, inp, dev, rank, world):
    from kimi_delta_attention_05_gb300 import kda as K
    import torch.distributed as dist
    steps = a.steps or DEFAULT_STEPS[a.workload]
    d, out, fin, args, ws = device_call(inp, dev)
    stream = torch.cuda.current_stream(dev)
    lib = K.load_library()
    import ctypes
    launches_per_step = lib.kda_fwd_launches(ctypes.byref(args))
    flush = L2Flush(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for trio in ev:
        for e in trio:
            e.record(stream)  # creates the underlying events
    torch.cuda.synchronize(dev)
    for _ in range(a.warmup):
        flush()
        K.kda_fwd_args_call(args, ws, stream)
    torch.cuda.synchronize(dev)
    handles = [[e.cuda_event for e in trio] for trio in ev]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        w0 = time.time()
        for i in range(steps):
            flush()  # untimed: outside this call's events
            K.kda_fwd_args_call(args, ws, stream, events=handles[i])
        torch.cuda.synchronize(dev)
        w1 = time.time()
    if world > 1:
        dist.barrier()
    chunk_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)]
    state_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(steps)]
    call_ms = [ev[i][0].elapsed_time(ev[i][2]) for i in range(steps)]  # one call, event to event
    ms = max_over_ranks(sum(call_ms), world, dev)  # the K timed calls, flushes excluded
    return dict(ms=ms, steps=steps, chunk_ms=statistics.mean(chunk_ms),
                state_ms=statistics.mean(state_ms), launches=launches_per_step * steps,
                call_median_ms=statistics.median(call_ms), call_min_ms=min(call_ms),
                clocks=clk.summary(w0, w1))


def run_e2e(a, inp, dev):
    """The public C-ABI call on HOST buffers (kda_fwd_host): every step copies
    the inputs from pinned host memory and the output (and final state) back
    inside the timed region; the library pipelines those copies with its
    kernels.  Returns (ms per step, H2D bytes, D2H bytes per step)."""
    from kimi_delta_attention_05_gb300.kda import host_device_bytes, kda_fwd_host_args_call, make_args
    host = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in inp.items()}
    names = ["q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state", "cu_seqlens"]
    h2d = sum(host[n].numel() * host[n].element_size() for n in names if host[n] is not None)
    stream = torch.cuda.current_stream(dev)
    H = inp["q"].shape[2]
    fin_dt = None if inp["final_state"] is None else (
        torch.bfloat16 if inp["final_state"] == "bf16" else torch.float32)
    out_host = torch.empty_like(inp["v"]).pin_memory()
    fin_host = None if fin_dt is None else torch.empty(
        (inp["N"], H, K_DIM, K_DIM), dtype=fin_dt).pin_memory()
    d2h = out_host.numel() * 2 + (0 if fin_host is None else fin_host.numel() * fin_host.element_size())
    lb = inp["lower_bound"] if inp["gate"] == "safe" else None
    args = make_args(host["q"], host["k"], host["v"], host["g"], host["beta"], inp["scale"],
                     out_host, host["A_log"], host["dt_bias"], lb, host["initial_state"], fin_host,
                     host["cu_seqlens"], inp["qk_l2norm"], inp["gate"])
    dbuf = torch.empty(max(host_device_bytes(args), 1), dtype=torch.uint8, device=dev)

    def step():
        kda_fwd_host_args_call(args, dbuf, stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    n = max(1, a.e2e_steps)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(n):
        step()
    s1.record(stream)
    torch.cuda.synchronize(dev)
    ms = s0.elapsed_time(s1) / n
    return ms, h2d, d2h


def oracle_sample(inp, budget_s):
    """Time the fp64 oracle on a bounded sample of (sequence, head) units."""
    import oracle
    H = inp["q"].shape[2]
    N = inp["N"]
    cu = inp["cu_seqlens"]
    lens = [int(cu[n + 1] - cu[n]) for n in range(N)] if cu is not None else [inp["q"].shape[1]] * N
    cores = len(os.sched_getaffinity(0))
    # calibrate on one small unit
    units_all = list(range(N * H))
    t0 = time.perf_counter()
    oracle.kda_recurrence(inp["q"][:, :256], inp["k"][:, :256], inp["v"][:, :256],
                          inp["g"][:, :256], inp["beta"][:, :256], scale=inp["scale"],
                          A_log=inp["A_log"], dt_bias=inp["dt_bias"],
                          lower_bound=inp["lower_bound"], gate=inp["gate"],
                          qk_l2norm=inp["qk_l2norm"], units=[0], threads=1)
    per_tok = (time.perf_counter() - t0) / 256
    budget_tok = budget_s * cores / max(per_tok, 1e-9)
    chosen, tok = [], 0
    step = max(1, len(units_all) // 64)
    for u in units_all[::step] + units_all:
        if u in chosen:
            continue
        if tok >= budget_tok:
            break
        chosen.append(u)
        tok += lens[u // H]
    t0 = time.perf_counter()
    oracle.kda_recurrence(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], scale=inp["scale"],
                          A_log=inp["A_log"], dt_bias=inp["dt_bias"],
                          lower_bound=inp["lower_bound"], gate=inp["gate"],
                          qk_l2norm=inp["qk_l2norm"], initial_state=inp["initial_state"],
                          cu_seqlens=cu, units=chosen, threads=cores)
    el = time.perf_counter() - t0
    sample_tokens = tok / H  # sequence tokens equivalent (heads not multiplied in)
    return dict(value=sample_tokens / el, unit="tokens/s", cores=cores, kind="oracle",
                sample=f"{len(chosen)} of {N * H} (sequence, head) units, {tok} token-heads, "
                       f"fp64 recurrence, {el:.1f} s wall")


def run_reference(a, inp):
    """Reference arm: the fp64 oracle as it stands, each step a bounded sample
    (one unit per host core) of the same workload."""
    import oracle
    H = inp["q"].shape[2]
    N = inp["N"]
    cu = inp["cu_seqlens"]
    lens = [int(cu[n + 1] - cu[n]) for n in range(N)] if cu is not None else [inp["q"].shape[1]] * N
    cores = len(os.sched_getaffinity(0))
    units = list(range(N * H))
    stride = max(1, len(units) // cores)
    chosen = units[::stride][:cores]
    tok = sum(lens[u // H] for u in chosen)
    steps = a.steps or 5

    def step():
        oracle.kda_recurrence(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              scale=inp["scale"], A_log=inp["A_log"], dt_bias=inp["dt_bias"],
                              lower_bound=inp["lower_bound"], gate=inp["gate"],
                              qk_l2norm=inp["qk_l2norm"], initial_state=inp["initial_state"],
                              cu_seqlens=cu, units=chosen, threads=cores)

    for _ in range(a.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    el = time.perf_counter() - t0
    value = steps * tok / H / el
    sample = (f"{len(chosen)} of {N * H} (sequence, head) units per step, {tok} token-heads, "
              f"fp64 recurrence")
    return dict(value=value, ms=el / steps * 1e3, steps=steps, cores=cores, sample=sample)


def workload_config(a, inp, world):
    w = WORKLOADS[a.workload]
    H = inp["q"].shape[2]
    total_bytes = sum(inp[n].numel() * inp[n].element_size()
                      for n in ("q", "k", "v", "g", "beta")) + inp["v"].numel() * 2
    cfg = {"workload": a.workload, "B": int(inp["q"].shape[0]), "T": int(inp["q"].shape[1]),
           "H": int(H), "K": K_DIM, "V": K_DIM, "N": int(inp["N"]), "gate": w.gate,
           "qk_l2norm": w.qk_l2norm, "initial_state": w.init_state, "final_state": w.final_state,
           "chunk": CHUNK, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
           "l2": f"inputs+outputs {total_bytes / 1e6:.0f} MB vs 129 MB L2; untimed L2 flush "
                 "between calls (256 MB written, another 256 MB read); each call timed by "
                 "its own CUDA events",
           "compute": "bf16 I/O; intra-chunk tcgen05 (bf16 A/P, fp16 WY; fp32 "
                      "tensor-memory accumulators) with 16x16 T blocks on mma.sync; state tcgen05 "
                      "(fp16 operands, fp32 tensor-memory accumulators); fp32 state"}
    return cfg


def run_recurrent_line(a, dev):
    """Decoding steps through kda_fwd_recurrent: the state stays on the device
    and is updated in place from step to step.  Compulsory bytes per step:
    the state read and written (fp32, 64 KiB each per (sequence, head)) plus
    the token inputs and outputs (1282 B per token-head)."""
    from kimi_delta_attention_05_gb300 import kda as K
    import ctypes
    name = "decode" if a.workload == "long_context" else a.workload
    inp = make_inputs(WORKLOADS[name])
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}
    state = d["initial_state"]
    out = torch.empty_like(d["v"])
    lb = inp["lower_bound"] if inp["gate"] == "safe" else None
    args = K.make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], out, d["A_log"],
                       d["dt_bias"], lb, state, state, d["cu_seqlens"], inp["qk_l2norm"],
                       inp["gate"])
    lib = K.load_library()
    stream = torch.cuda.current_stream(dev)
    call = lambda: lib.kda_fwd_recurrent(ctypes.byref(args), ctypes.c_void_p(stream.cuda_stream))
    steps = a.steps or 2000
    for _ in range(a.warmup):
        assert call() == 0
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        w0 = time.time()
        t0.record(stream)
        for _ in range(steps):
            call()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        w1 = time.time()
    ms_step = t0.elapsed_time(t1) / steps
    th = token_heads(inp)
    H = inp["q"].shape[2]
    tokens = th // H
    units = inp["N"] * H
    state_bytes = 2 * units * K_DIM * K_DIM * state.element_size()
    step_bytes = state_bytes + th * (BYTES_IN_PER_TOKEN_HEAD + BYTES_OUT_PER_TOKEN_HEAD)
    hbm, _, peak_kind = measured_peaks()
    achieved = step_bytes / (ms_step * 1e-3) / 1e9
    # fp32 arithmetic against the CUDA cores' peak (SM count x 128 FMA lanes x 2
    # flop x the maximum SM clock): the launches issue fp32 multiply-adds
    if inp["cu_seqlens"] is not None:
        cu = inp["cu_seqlens"].tolist()
        chunks = sum((cu[i + 1] - cu[i] + 63) // 64 for i in range(len(cu) - 1))
    else:
        chunks = int(inp["q"].shape[0]) * ((int(inp["q"].shape[1]) + 63) // 64)
    fma_item = bwd_fma_per_chunk_head()
    flops = 2.0 * fma_item * chunks * H
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = sm_max_mhz()
    fp32_peak = sms * 128 * 2 * mhz * 1e6 / 1e12
    # end to end: token inputs H2D from pinned memory and outputs D2H each step,
    # the state resident on the device (a serving loop's traffic)
    names = ["q", "k", "v", "g", "beta"]
    host = {n: inp[n].pin_memory() for n in names}
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e_steps = max(a.e2e_steps, 1)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e_steps):
        for n in names:
            d[n].copy_(host[n], non_blocking=True)
        call()
        host_out.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e_ms = e0.elapsed_time(e1) / e_steps
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = host_out.numel() * host_out.element_size()
    cfg = {"workload": name, "B": int(inp["q"].shape[0]), "T": int(inp["q"].shape[1]), "H": int(H),
           "K": K_DIM, "V": K_DIM, "N": int(inp["N"]), "gate": inp["gate"],
           "qk_l2norm": bool(inp["qk_l2norm"]), "state": "fp32, updated in place",
           "path": "token-by-token (kda_fwd_recurrent)", "parallelism": "single GPU",
           "l2": f"state {state_bytes // 2 / 1e6:.0f} MB > 129 MB L2; no flush"}
    line = {"metric": "KDA decode tokens/s and % of HBM roofline, 1 GB300", "value": tokens / (ms_step * 1e-3),
            "unit": "tokens/s", "n_gpus": 1, "steps": steps, "warmup": a.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": cfg,
            "roofline": {"bound": "hbm", "kernel": "kda_recurrent_kernel", "achieved": achieved,
                         "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": recorded_traffic("kda_recurrent_kernel", name),
                         "algorithmic_bytes_per_launch": step_bytes,
                         "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})"},
            "gpu_launches": steps, "clocks": clk.summary(w0, w1),
            "e2e": {"value": tokens / (e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}}
    print(json.dumps(line), flush=True)
    return 0


# backward bytes per token-head: q, k, v, g, dout (bf16) and beta in; dq, dk,
# dv, dg (fp32) and dbeta (fp32) out
BWD_BYTES_PER_TOKEN_HEAD = 5 * 2 * K_DIM + 2 + 4 * 4 * K_DIM + 4


def bwd_fma_per_chunk_head(C=64, D=K_DIM):
    """fp32 multiply-adds of the chunked backward per (64-token chunk, head),
    as it is formulated (dense C x C factors, padded chunks): recompute, the two
    state chains, the gradient products and the chunk gradients."""
    prep = (4 * 136 * D * 2                                  # G, P inside the 16-token blocks
            + sum(16 * 16 * i * D * 2 for i in (1, 2, 3))    # G, P left of the diagonal blocks
            + 4 * 16 * 120 + sum((4 - d) * 256 * (16 * d + 16) for d in (1, 2, 3))  # (I+A)^-1
            + 2 * C * C * D)                                 # W, U
    fwd = 2 * C * D * D                                      # U - W S^T, U_new^T Khat
    rev = C * D * (D + C) + 2 * D * D * C                    # dU; dS
    prod = 3 * C * D * D + 2 * C * C * D + C * C * D + 2 * C * D * C + D * D  # dQg dW dKhat; dT; dP; dV dKg; dgC
    grad = (2 * C ** 3 + 4 * 16 * 15 * D * 4                  # dM; pairwise inside the blocks
            + 2 * sum(16 * 16 * i * D * 2 for i in (1, 2, 3)) + C * D * 6)  # left of the blocks; scalings
    return prep + fwd + rev + prod + grad


def run_backward_line(a, dev):
    """kda_bwd on the workload: gradients of <out, dout> (+ <final, dfinal>
    when the workload has a final state) with respect to every input.  Each
    call is timed by its own events (kda_bwd_profiled: prep and forward state
    pass, reverse state pass, chunk gradients and finalize), with an untimed L2
    flush between calls."""
    from kimi_delta_attention_05_gb300 import kda as K
    w = WORKLOADS[a.workload]
    inp = make_inputs(w)
    gen = torch.Generator().manual_seed(w.seed + 1000)
    dout_h = torch.randn(inp["v"].shape, generator=gen).to(torch.bfloat16)
    H = inp["q"].shape[2]
    dfin_h = (torch.randn((inp["N"], H, K_DIM, K_DIM), generator=gen)
              if inp["final_state"] is not None else None)
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}
    dout = dout_h.to(dev)
    dfin = dfin_h.to(dev) if dfin_h is not None else None
    lb = inp["lower_bound"] if inp["gate"] == "safe" else None
    args, grads = K.make_bwd_args(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], dout,
                                  d["A_log"], d["dt_bias"], lb, d["initial_state"], dfin,
                                  d["cu_seqlens"], qk_l2norm=inp["qk_l2norm"], gate=inp["gate"])
    ws = torch.empty(max(K.bwd_workspace_bytes(args), 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    steps = a.steps or 20
    flush = L2Flush(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for quad in ev:
        for e in quad:
            e.record(stream)
    for _ in range(a.warmup):
        flush()
        K.kda_bwd_args_call(args, ws, stream)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        w0 = time.time()
        for i in range(steps):
            flush()
            K.kda_bwd_args_call(args, ws, stream, events=[e.cuda_event for e in ev[i]])
        torch.cuda.synchronize(dev)
        w1 = time.time()
    stage = {name: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps))
             for j, name in enumerate(["prep + forward state pass", "reverse state pass",
                                       "gradient products + chunk gradients + finalize"])}
    ms_step = statistics.mean(ev[i][0].elapsed_time(ev[i][3]) for i in range(steps))
    th = token_heads(inp)
    tokens = th // H
    units = inp["N"] * H
    st_bytes = 0
    if inp["initial_state"] is not None:
        st_bytes += 2 * units * K_DIM * K_DIM * inp["initial_state"].element_size() + units * K_DIM * K_DIM * 4
    if dfin is not None:
        st_bytes += units * K_DIM * K_DIM * 4
    step_bytes = th * BWD_BYTES_PER_TOKEN_HEAD + st_bytes
    hbm, _, peak_kind = measured_peaks()
    achieved = step_bytes / (ms_step * 1e-3) / 1e9
    # fp32 arithmetic against the CUDA cores' peak (SM count x 128 FMA lanes x 2
    # flop x the maximum SM clock): the launches issue fp32 multiply-adds
    if inp["cu_seqlens"] is not None:
        cu = inp["cu_seqlens"].tolist()
        chunks = sum((cu[i + 1] - cu[i] + 63) // 64 for i in range(len(cu) - 1))
    else:
        chunks = int(inp["q"].shape[0]) * ((int(inp["q"].shape[1]) + 63) // 64)
    fma_item = bwd_fma_per_chunk_head()
    flops = 2.0 * fma_item * chunks * H
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = sm_max_mhz()
    fp32_peak = sms * 128 * 2 * mhz * 1e6 / 1e12
    # end to end: inputs and dout in from pinned host memory, token gradients
    # back, around the same call
    names = ["q", "k", "v", "g", "beta"]
    host = {n: inp[n].pin_memory() for n in names}
    host_dout = dout_h.pin_memory()
    host_g = {n: torch.empty(grads[n].shape, dtype=torch.float32).pin_memory()
              for n in ["q", "k", "v", "g", "beta"]}
    e_steps = max(min(a.e2e_steps, 10), 1)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e_steps):
        for n in names:
            d[n].copy_(host[n], non_blocking=True)
        dout.copy_(host_dout, non_blocking=True)
        K.kda_bwd_args_call(args, ws, stream)
        for n, t in host_g.items():
            t.copy_(grads[n], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e_ms = e0.elapsed_time(e1) / e_steps
    h2d = sum(host[n].numel() * host[n].element_size() for n in names) + host_dout.numel() * 2
    d2h = sum(t.numel() * 4 for t in host_g.values())
    cfg = {"workload": a.workload, "B": int(inp["q"].shape[0]), "T": int(inp["q"].shape[1]),
           "H": int(H), "K": K_DIM, "V": K_DIM, "N": int(inp["N"]), "gate": inp["gate"],
           "qk_l2norm": bool(inp["qk_l2norm"]), "initial_state": w.init_state,
           "dfinal_state": "fp32" if dfin is not None else None,
           "path": "backward (kda_bwd): chunked WY form in fp32 on the CUDA cores; per 64-token chunk "
                   "recompute, forward and reverse state passes (16 value rows per CTA), gradient "
                   "products and chunk gradients",
           "parallelism": "single GPU",
           "l2": "untimed L2 flush between calls (256 MB written, another 256 MB read); each call "
                 "timed by its own CUDA events"}
    dom = max(stage, key=stage.get)
    # prep, forward pass, reverse pass, products, gradients; finalize with gate
    # parameters; the chunk prefix with packed sequences
    launches = 5 + (1 if (grads["A_log"] is not None or grads["dt_bias"] is not None) else 0) \
        + (1 if inp["cu_seqlens"] is not None else 0)
    line = {"metric": "KDA bwd tokens/s and % of HBM roofline, 1 GB300", "value": tokens / (ms_step * 1e-3),
            "unit": "tokens/s", "n_gpus": 1, "steps": steps, "warmup": a.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": cfg,
            "roofline": {"bound": "alu", "kernel": f"kda_bwd ({launches} launches)",
                         "achieved": flops / (ms_step * 1e-3) / 1e12, "peak": fp32_peak, "unit": "TFLOP/s",
                         "frac": flops / (ms_step * 1e-3) / 1e12 / fp32_peak, "traffic": None,
                         "fp32_fma_per_chunk_head": fma_item, "chunk_heads": chunks * H,
                         "dominant_launch": dom,
                         "peak_source": f"{sms} SMs x 128 fp32 FMA lanes x 2 flop x {mhz:.0f} MHz (unit counts, maximum clock)",
                         "hbm": {"achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                                 "algorithmic_bytes_per_call": step_bytes,
                                 "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})"}},
            "stages_ms": stage, "gpu_launches": launches * steps, "clocks": clk.summary(w0, w1),
            "e2e": {"value": tokens / (e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    a = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = WORKLOADS[a.workload]

    if a.impl == "reference":
        if rank != 0:
            return 0
        inp = make_inputs(w)
        r = run_reference(a, inp)
        line = {"impl": "reference", "metric": METRIC, "value": r["value"], "unit": "tokens/s",
                "n_gpus": a.gpus, "steps": r["steps"], "warmup": a.warmup, "ms_per_step": r["ms"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": workload_config(a, inp, 1),
                "cpu_baseline": {"value": r["value"], "unit": "tokens/s", "cores": r["cores"],
                                 "kind": "oracle", "sample": r["sample"]},
                "e2e": {"value": r["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from kimi_delta_attention_05_gb300 import kda as K
    K.load_library()
    if a.path == "recurrent":
        return run_recurrent_line(a, dev) if rank == 0 else 0
    if a.path == "backward":
        return run_backward_line(a, dev) if rank == 0 else 0
    inp = rank_inputs(w, rank)
    r = run_ours(a, inp, dev, rank, world)
    th = token_heads(inp)
    H = inp["q"].shape[2]
    tokens = th // H
    ms_step = r["ms"] / r["steps"]
    value = whole_job_value(tokens, world, ms_step)
    hbm, bf16, peak_kind = measured_peaks()
    sio = state_io_bytes(inp)
    chunk_bytes = th * BYTES_IN_PER_TOKEN_HEAD
    state_bytes = th * BYTES_OUT_PER_TOKEN_HEAD + sio
    dom = "kda_chunk_kernel" if r["chunk_ms"] >= r["state_ms"] else "kda_state_kernel"
    dom_ms = max(r["chunk_ms"], r["state_ms"])
    dom_bytes = chunk_bytes if dom == "kda_chunk_kernel" else state_bytes
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    path_bytes = chunk_bytes + state_bytes
    path_gbs = path_bytes / (ms_step * 1e-3) / 1e9
    flops = th * FLOP_PER_TOKEN_HEAD
    roof_t = max(flops / (bf16 * 1e12), path_bytes / (hbm * 1e9))
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": r["steps"],
        "warmup": a.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(a, inp, world),
        "tflops": flops / (ms_step * 1e-3) / 1e12,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": recorded_traffic(dom, a.workload),
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
                     "path": {"achieved": path_gbs, "frac": path_gbs / hbm,
                              "roofline_ms": roof_t * 1e3, "frac_of_roofline": roof_t * 1e3 / ms_step}},
        "stages_ms": {"kda_chunk_kernel": r["chunk_ms"], "kda_state_kernel": r["state_ms"]},
        "call_ms": {"median": r["call_median_ms"], "min": r["call_min_ms"],
                    "note": "per call, from the event before its first launch to the one after its last"},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    lpc = r["launches"] // r["steps"]
    line["config"]["state_pass"] = ("sequence split: segment runs, transition chain, re-runs "
                                    "(4 launches per call)" if lpc == 4 else f"one pass ({lpc} launches per call)")
    if rank == 0:
        e_ms, h2d, d2h = run_e2e(a, inp, dev)
        line["e2e"] = {"value": tokens * world / (e_ms * 1e-3), "unit": "tokens/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}
        if world == 1 and not a.no_cpu_baseline:
            line["cpu_baseline"] = oracle_sample(inp, a.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
