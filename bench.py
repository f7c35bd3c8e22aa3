"""Benchmark: credit-assignment timesteps/s of GAE with truncation bootstrapping on
[4096, 1024] fp32 rollouts, and the fraction of the GB300 HBM roofline it reaches.

One step = one fused GAE launch (load -> operand build -> segmented reverse scan ->
advantages and returns written once) over one [4096, 1024] batch that is already in
HBM. Batches rotate over several distinct seeded input sets whose total size exceeds
the L2 cache, so no step reads another step's inputs from L2. The timed steps are
replayed from CUDA graphs so that host launch overhead does not idle the GPU.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl rlca|reference]
With --impl reference the fp64 CPU oracle is timed instead, on a bounded sample of the
same workload, on this host's cores. Under torchrun every rank runs its own batch
(weak scaling, no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic_rollouts as sr  # noqa: E402

METRIC = "credit-assignment timesteps/sec at [4096,1024] fp32; % of GB300 HBM roofline"
UNIT = "timesteps/s"
N_ENVS, SEQ_LEN = 4096, 1024
WORKLOAD = "GAE with truncation bootstrapping, fp32, num_envs=4096, seq_len=1024"
WORKLOADS = {
    "gae": WORKLOAD,
    "return": "discounted return, fp32, num_envs=4096, seq_len=1024 (rates of the [4096,128] return/TD workload)",
    "td_lambda": "TD(lambda=0.9), fp32, num_envs=4096, seq_len=1024 (rates of the [4096,128] return/TD workload)",
    "vtrace": "V-trace, fp32, num_envs=4096, seq_len=1024 (rates of the [8192,256] V-trace workload)",
    "retrace": "Retrace, fp32, num_envs=4096, seq_len=1024 (rates of the [2048,4096] Retrace workload)",
    "td_multi": "TD(lambda) for lambda in {0, 0.9, 1} fused, fp32, num_envs=4096, seq_len=1024",
    "gae_vtrace": "GAE (lambda=0.95) and V-trace fused, fp32, num_envs=4096, seq_len=1024 "
                  "(rates of the [8192,256] V-trace workload)",
    "gae_bf16": "GAE with truncation bootstrapping, bf16 inputs / fp32 math and outputs, "
                "num_envs=4096, seq_len=1024",
    "trace": "eligibility trace (forward scan), fp32, num_envs=4096, seq_len=1024",
    "prefix_sum": "episodic prefix sum (forward scan), fp32, num_envs=4096, seq_len=1024",
}
for _e in ("return", "td_lambda", "vtrace", "retrace", "trace", "prefix_sum"):
    WORKLOADS[_e + "_bf16"] = WORKLOADS[_e].replace(", fp32,", ", bf16 inputs / fp32 math and "
                                                    "outputs,")
for _e in ("gae", "return", "td_lambda", "vtrace", "retrace", "trace", "prefix_sum"):
    WORKLOADS[_e + "_fp16"] = WORKLOADS[_e].replace(", fp32,", ", fp16 inputs / fp32 math and "
                                                    "outputs,")
_EST_NAME = {"gae": "GAE", "return": "return", "td_lambda": "TD(lambda)", "vtrace": "V-trace",
             "retrace": "Retrace"}

# Estimators with a 16-bit-input variant: "<base>_bf16" / "<base>_fp16" runs the base
# estimator's _bf16 / _fp16 entry point on the same workload, its per-step data inputs
# rounded to that format.
NARROW = {"_bf16": "bfloat16", "_fp16": "float16"}


def base_est(est: str) -> str:
    """The estimator an entry of the bench computes, without its input-format suffix."""
    for suffix in NARROW:
        if est.endswith(suffix):
            return est[:-len(suffix)]
    return est


def data_dtype_of(torch, est: str):
    """Torch dtype of the per-step data inputs for `est` (None = fp32)."""
    for suffix, name in NARROW.items():
        if est.endswith(suffix):
            return getattr(torch, name)
    return None


def kernel_desc(est: str, N: int, T: int, workspace: bool, sms: int) -> str:
    """The kernel the library's dispatch picks for this call (contiguous rows)."""
    be = base_est(est)
    narrow = be != est
    if be in ("trace", "prefix_sum"):
        if T <= 256:
            return "credit_forward_kernel (warp-owned rows, forward)"
        ctas = (N + 3) // 4
        depth = 3 if narrow or 9 * sms <= 2 * ctas <= 14 * sms else 2
        return (f"credit_forward_pipe_kernel (a warp per row walking forward, {depth} chunks "
                "of loads in flight)" if T <= 1024
                else "credit_forward_tile_kernel (CTA row loop, forward)")
    if be == "td_multi":
        if T <= 256:
            return "credit_td_multi_warp_kernel (warp-owned rows, 3 lambdas per load)"
        if T <= 512:
            return "credit_td_multi_kernel (whole-row CTA tiles, 3 lambdas per load)"
        return ("credit_td_multi_pipe_kernel (a warp per row, next chunk's loads in flight, "
                "3 lambdas per load)" if T <= 1024
                else "credit_td_multi_kernel (CTA row loop, 3 lambdas per load)")
    if be == "gae_vtrace":
        return ("credit_gae_vtrace_kernel (CTA tiles, GAE and V-trace per load)" if T <= 1024
                else "credit_gae_vtrace_kernel (CTA row loop, GAE and V-trace per load)")
    name = _EST_NAME[be] + (f", {est[len(be) + 1:]} inputs" if narrow else "")
    if narrow:
        if T <= 256:
            return f"credit_warp_kernel<{name}> (warp-owned rows, 8 steps/lane)"
        pipe_from = 256 if be == "gae" else (1024 if be == "return" else 512)
        depth = 1 if be in ("vtrace", "retrace") else 2
        if pipe_from < T <= 1024:
            return (f"credit_warp_pipe_kernel<{name}> (a warp per row, {depth} chunk(s) of "
                    "loads in flight)")
        if be == "gae":
            return f"credit_warp_kernel<{name}> (warp-owned rows, 16 steps/lane)"
        return (f"credit_scan_kernel<{name}, whole-row CTA tiles>" if T <= 1024
                else f"credit_scan_kernel<{name}, CTA row loop>")
    if T > 1024:
        if workspace and N < 2 * sms:
            return f"credit_scan_kernel<{name}, look-back across CTA tiles>"
        return f"credit_scan_kernel<{name}, CTA row loop>"
    if (T in (64, 128, 256) and N % (256 // T) == 0 and be in ("return", "td_lambda", "gae")
            and N * T > 4096 * 256):
        rows = "the rows" if T == 256 else f"blocks of {256 // T} rows"
        return (f"credit_warp_rows_pipe_kernel<{name}> (one wave of warps walking {rows}, "
                "the next block's loads in flight)")
    if T <= 256:
        return f"credit_warp_kernel<{name}> (warp-owned rows)"
    if be == "return" and 512 < T <= 960 and (N + 3) // 4 <= 7 * sms:
        return (f"credit_warp_pipe_kernel<{name}> (a warp per row, 2 chunks of loads in "
                "flight, 7 CTAs per SM)")
    if be == "gae" or (be == "td_lambda" and T > 512):
        return f"credit_warp_pipe_kernel<{name}> (a warp per row, next chunk's loads in flight)"
    return f"credit_scan_kernel<{name}, whole-row CTA tiles>"


FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20

# Traffic per launch measured by ncu (one captured launch, --set full, the commands in
# the committed ncu summaries): dram__bytes_read.sum + 32 x
# lts__t_sectors_srcunit_tex_op_write.sum (within one captured launch the outputs stay
# in L2, so the DRAM write counter misses them; the L2 write sectors count what the SMs
# wrote, partial sectors included). Keyed by (hash of the kernel sources at the time of
# the capture, estimator, N, T, workspace); null once the kernels change.
_H = "208d2a2360ac377f"
NCU_TRAFFIC = {
    (_H, "gae", 4096, 1024, False): 80_551_296,
    (_H, "return", 4096, 1024, False): 37_773_568,
    (_H, "td_lambda", 4096, 1024, False): 55_704_320,
    (_H, "vtrace", 4096, 1024, False): 88_113_152,
    (_H, "retrace", 4096, 1024, False): 88_111_872,
    (_H, "td_multi", 4096, 1024, False): 92_466_432,
    (_H, "gae_vtrace", 4096, 1024, False): 121_673_728,
    (_H, "trace", 4096, 1024, False): 44_281_728,
    (_H, "gae_bf16", 4096, 1024, False): 63_315_072,
    (_H, "gae_fp16", 4096, 1024, False): 62_731_648,
    (_H, "return_bf16", 4096, 1024, False): 29_385_472,
    (_H, "vtrace_fp16", 4096, 1024, False): 64_391_808,
    (_H, "retrace", 2048, 4096, False): 176_225_536,
    (_H, "return", 4096, 128, False): 4_750_336,
    (_H, "vtrace", 8192, 256, False): 44_100_352,
    (_H, "gae", 8192, 256, False): 38_320_128,
    (_H, "return", 16384, 128, False): 18_953_216,
    (_H, "return", 16, 524288, True): 76_033_824,
    (_H, "td_multi", 4096, 128, False): 11_047_168,
    (_H, "td_lambda", 4096, 128, False): 6_850_560,
    (_H, "gae", 16, 128, False): 61_952,
    (_H, "trace", 4096, 128, False): 5_275_904,
    (_H, "td_lambda_bf16", 4096, 1024, False): 38_164_864,
    (_H, "retrace_bf16", 4096, 1024, False): 56_016_512,
    (_H, "trace_bf16", 4096, 1024, False): 35_073_152,
    (_H, "return", 4096, 600, False): 22_976_448,
    (_H, "trace_fp16", 4096, 1024, False): 35_061_376,
    (_H, "trace", 8192, 1024, False): 85_687_808,
}


def kernel_source_hash() -> str:
    """Hash of the code that decides which kernel runs and what it does: the device code
    and launch logic (csrc/*.cuh and the kernel units, csrc/*.cu but the C-ABI files),
    with comments and blank lines removed so that editing a comment keeps the recorded
    traffic. The C-ABI validation (api.cu, noalloc.cu) and the measurement copy
    (measure.cu) launch no estimator kernel themselves and are left out."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "segmented_associative_scan_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith(".cuh") or (name.endswith(".cu") and
                                     name not in ("api.cu", "noalloc.cu", "measure.cu")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                text = f.read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            text = re.sub(r"//[^\n]*", "", text)
            code = "\n".join(l.rstrip() for l in text.splitlines() if l.strip())
            h.update(name.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)"


# Per-step data input arrays and output arrays of each estimator entry.
N_DATA_INPUTS = {"return": 1, "td_lambda": 2, "gae": 2, "vtrace": 3, "retrace": 4, "trace": 1,
                 "prefix_sum": 1, "td_multi": 2, "gae_vtrace": 3}
N_OUTPUTS = {"return": 1, "td_lambda": 1, "gae": 2, "vtrace": 2, "retrace": 1, "trace": 1,
             "prefix_sum": 1, "td_multi": 3, "gae_vtrace": 4}


def algorithmic_bytes(est: str, ro) -> int:
    """Minimal HBM bytes of one launch: every input element the estimator needs read once
    (truncation values only where a step is truncated and not terminated; per-env
    bootstrap values once) and every output written once."""
    n = ro.N * ro.T
    be = base_est(est)
    in_bytes = 4 if be == est else 2
    b = n * (in_bytes * N_DATA_INPUTS[be] + 1 + 4 * N_OUTPUTS[be])
    if ro.truncated is not None:
        b += n
        if be not in ("trace", "prefix_sum"):  # forward scans read no truncation values
            b += in_bytes * int(np.count_nonzero(ro.truncated & (1 - ro.terminated)))
    if ro.bootstrap is not None:
        b += 4 * ro.N
    return b


def workload_inputs(est: str, N: int, T: int, seed: int):
    """The seeded workload each estimator is quoted on, at [N, T]."""
    est = base_est(est)
    if est == "gae":
        return sr.gae_trunc(N=N, T=T, seed=seed)
    if est in ("trace", "prefix_sum"):
        return sr.traces(N=N, T=T, seed=seed)
    if est in ("return", "td_lambda", "td_multi"):
        return sr.return_td(N=N, T=T, seed=seed)
    if est in ("vtrace", "gae_vtrace"):
        return sr.vtrace(N=N, T=T, seed=seed)
    return sr.retrace(N=N, T=T, seed=seed)


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons every 100 ms, in the
    background; `summary(t0, t1)` keeps the samples taken inside [t0, t1]."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                self.samples.append(dict(t=time.time(), sm=float(parts[2]),
                                         sm_max=float(parts[3]),
                                         reasons=[name for name, v in zip(
                                             ("hw_slowdown", "hw_thermal_slowdown",
                                              "sw_thermal_slowdown", "sw_power_cap"),
                                             parts[5:9]) if v.lower() == "active"]))
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s["t"] <= t1]
        window = "timed region"
        if not inside:
            inside = self.samples
            window = "whole run (timed region shorter than the 100 ms sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "nvidia-smi unavailable"}
        reasons = sorted({r for s in inside for r in s["reasons"]})
        return {"sm_mhz": statistics.median(s["sm"] for s in inside),
                "sm_max_mhz": max(s["sm_max"] for s in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


# --------------------------------------------------------------------------- ranks

def max_over_ranks(value: float, dist) -> float:
    """The largest `value` over all ranks (host-side timing only; the data path has no
    collective). NCCL reduces a CUDA tensor, gloo a CPU one."""
    if dist is None:
        return value
    import torch
    on_gpu = dist.get_backend() == "nccl"
    dev = torch.device("cuda", torch.cuda.current_device()) if on_gpu else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, N: int, T: int, steps: int, ms_max: float) -> float:
    """Whole-job timesteps/s: every rank processed its own batch each step (weak
    scaling), and the job took as long as its slowest rank."""
    return world * N * T * steps / (ms_max * 1e-3)


# --------------------------------------------------------------------------- GPU arm

class DeviceSet:
    """One batch resident in HBM plus its output buffers (data inputs in `data_dtype`)."""

    def __init__(self, ro, device, data_dtype=None):
        import torch
        self.ro = ro

        def t(a):
            if a is None:
                return None
            x = torch.from_numpy(a).to(device)
            return x.to(data_dtype) if data_dtype is not None and x.is_floating_point() \
                and x.dim() == 2 else x
        self.reward, self.value = t(ro.reward), t(ro.value)
        self.terminated, self.truncated = t(ro.terminated), t(ro.truncated)
        self.trunc_value, self.bootstrap = t(ro.trunc_value), t(ro.bootstrap)
        self.log_rho, self.q_taken, self.expected_q, self.rho = (
            t(ro.log_rho), t(ro.q_taken), t(ro.expected_q), t(ro.rho))
        z = lambda: torch.empty((ro.N, ro.T), dtype=torch.float32, device=device)
        self.out0, self.out1, self.out2, self.out3 = z(), z(), z(), z()
        self.ws = None  # look-back workspace (the _ex entry points), when asked for

    def clone(self):
        import torch
        c = object.__new__(DeviceSet)
        for k, v in self.__dict__.items():
            setattr(c, k, v.clone() if isinstance(v, torch.Tensor) else v)
        return c


def launch(rlca, est, s, params):
    est = base_est(est)  # the binding picks the _bf16 entry point from the tensors' dtype
    fl = dict(terminated=s.terminated, truncated=s.truncated,
              trunc_value=s.trunc_value if s.truncated is not None else None)
    g = params["gamma"]
    ws = s.ws
    if est == "gae":
        rlca.rlca_gae(s.reward, s.value, **fl, bootstrap=s.bootstrap, gamma=g,
                      lam=params["lam"], advantages=s.out0, returns=s.out1, workspace=ws)
    elif est == "return":
        rlca.rlca_discounted_return(s.reward, **fl, bootstrap=s.bootstrap, gamma=g,
                                    returns=s.out0, workspace=ws)
    elif est == "td_lambda":
        rlca.rlca_td_lambda(s.reward, s.value, **fl, bootstrap=s.bootstrap, gamma=g,
                            lam=params["lam"], targets=s.out0, workspace=ws)
    elif est == "vtrace":
        rlca.rlca_vtrace(s.reward, s.value, s.log_rho, **fl, bootstrap=s.bootstrap, gamma=g,
                         lam=params["lam"], rho_bar=params["rho_bar"],
                         c_bar=params["c_bar"], pg_rho_bar=params["pg_rho_bar"],
                         vs=s.out0, pg_advantages=s.out1, workspace=ws)
    elif est == "retrace":
        rlca.rlca_retrace(s.reward, s.q_taken, s.expected_q, s.rho, **fl,
                          bootstrap_ev=s.bootstrap, gamma=g, lam=params["lam"], q_ret=s.out0,
                          workspace=ws)
    elif est == "gae_vtrace":
        rlca.rlca_gae_vtrace(s.reward, s.value, s.log_rho, **fl, bootstrap=s.bootstrap, gamma=g,
                             lam=0.95, lam_vtrace=params["lam"], rho_bar=params["rho_bar"],
                             c_bar=params["c_bar"], pg_rho_bar=params["pg_rho_bar"],
                             advantages=s.out0, returns=s.out1, vs=s.out2,
                             pg_advantages=s.out3)
    elif est == "td_multi":
        rlca.rlca_td_lambda_multi(s.reward, s.value, **fl, bootstrap=s.bootstrap, gamma=g,
                                  lams=params["lams"], targets=[s.out0, s.out1, s.out2])
    elif est == "trace":
        rlca.rlca_eligibility_trace(s.value, s.terminated, s.truncated, s.bootstrap,
                                    decay=params["decay"], traces=s.out0)
    else:
        rlca.rlca_episodic_prefix_sum(s.value, s.terminated, s.truncated, s.bootstrap,
                                      sums=s.out0)


def est_params(est, ro):
    p = dict(ro.params)
    if base_est(est) == "td_lambda":
        p["lam"] = 0.9
    return p


def capture(torch, step, n_sets, n_steps, first=0):
    """A CUDA graph of n_steps calls step(i), i = (first + k) % n_sets."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for k in range(n_steps):
            step((first + k) % n_sets)
    return g


def timed_replay(torch, graphs, lead):
    """Replay graphs between two CUDA events on the current stream; ms elapsed.

    `lead`, an untimed graph, is replayed first: while the GPU runs it, the host submits
    the start event and the timed graphs, so the timed region starts with work already
    queued and holds exactly the launches of `graphs` (their submission latency stays
    outside the events)."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    lead.replay()
    e0.record()
    for g in graphs:
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def n_sets_for(bytes_per_set):
    """Input sets to rotate so that their total exceeds the L2 cache 2.5 times (at most
    64 sets; tiny problems then stay L2-resident, which the config line states)."""
    return min(64, max(3, int(np.ceil(2.5 * L2_BYTES / bytes_per_set))))


def us_per_step(torch, step, n_sets, launches=300):
    """Average µs of step(i) over about `launches` back-to-back calls cycling the sets,
    replayed from a CUDA graph after a warm-up."""
    for i in range(3):
        step(i % n_sets)
    G = 10 * n_sets
    g = capture(torch, step, n_sets, G)
    g.replay()
    reps = max(1, launches // G)
    ms = timed_replay(torch, [g] * reps, g)
    return 1000.0 * ms / (G * reps)


def copy_pattern(est, s):
    """The arrays of set `s` that a plain copy with `est`'s byte pattern streams: the
    estimator's fp32 data inputs, its flag arrays and its outputs."""
    be = base_est(est)
    ins = {"return": [s.reward], "td_lambda": [s.reward, s.value], "gae": [s.reward, s.value],
           "td_multi": [s.reward, s.value], "vtrace": [s.reward, s.value, s.log_rho],
           "gae_vtrace": [s.reward, s.value, s.log_rho],
           "retrace": [s.reward, s.q_taken, s.expected_q, s.rho],
           "trace": [s.value], "prefix_sum": [s.value]}[be]
    flags = [s.terminated] + ([s.truncated] if s.truncated is not None else [])
    outs = [s.out0, s.out1, s.out2, s.out3][:N_OUTPUTS[be]]
    return ins, flags, outs


def warp_walk_chunks(est, T):
    """256-step chunks a warp walks in the kernel the dispatch picks for `est` at T (the
    pipelined warp rows), else 1 (warp-owned rows, CTA tiles)."""
    be = base_est(est)
    if be != est:  # 16-bit inputs: GAE and the forward scans from 257 steps, the rest
        walks = (256 < T <= 1024 if be in ("gae", "trace", "prefix_sum")  # from 513, but
                 else be != "return" and 512 < T <= 1024)               # not the return
    else:
        walks = ((be in ("gae", "trace", "prefix_sum") and 256 < T <= 1024)
                 or (be in ("td_multi", "td_lambda") and 512 < T <= 1024))
    chunks = -(-T // 256) if walks else 1
    return chunks if chunks in (1, 2, 4) else 1  # the copy takes 1, 2 or 4


def time_workload(torch, rlca, device, peak, est, ro, ceiling=True):
    """One estimator alone on the batch `ro` (copies of it rotating past L2 when it is
    large enough): µs per launch, achieved GB/s and the roofline fractions; with
    `ceiling`, also the best plain copy of the same bytes (rlca_measure_copy)."""
    params = est_params(est, ro)
    nbytes = algorithmic_bytes(est, ro)
    base = DeviceSet(ro, device, data_dtype_of(torch, est))
    n_sets = n_sets_for(nbytes)
    sets = [base] + [base.clone() for _ in range(n_sets - 1)]
    us = us_per_step(torch, lambda i: launch(rlca, est, sets[i], params), n_sets)
    gbs = nbytes / (us * 1e-6) / 1e9
    out = {"us_per_launch": round(us, 3), "algorithmic_bytes": nbytes,
           "bytes_per_step": round(nbytes / (ro.N * ro.T), 3),
           "achieved_gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
           "frac_of_8tbs": round(gbs / 8000.0, 4),
           "timesteps_per_s": round(ro.N * ro.T / (us * 1e-6), 1),
           "inputs_exceed_l2": n_sets * nbytes > L2_BYTES}
    traffic = NCU_TRAFFIC.get((kernel_source_hash(), est, ro.N, ro.T, False))
    if traffic is not None:  # bytes one captured launch moved, against the algorithmic
        out["ncu_traffic_ratio"] = round(traffic / nbytes, 3)
    if ceiling:
        # The best plain copy of the same bytes: in the kernel's launch shape, and for a
        # kernel that walks rows per warp also in the flat shape (one chunk per warp).
        pats = [copy_pattern(est, x) for x in sets]
        walk = warp_walk_chunks(est, ro.T)
        shapes = {}
        for chunks in sorted({1, walk}):
            shapes[chunks] = us_per_step(
                torch, lambda i: rlca.measure_copy(*pats[i], chunks=chunks), n_sets)
        best = min(shapes, key=shapes.get)
        out["ceiling_us"] = round(shapes[best], 3)
        out["ceiling_chunks_per_warp"] = best
        out["frac_of_ceiling"] = round(shapes[best] / us, 4)
    del sets, base
    torch.cuda.empty_cache()
    return out


ESTIMATORS_1024 = ("return", "td_lambda", "gae", "vtrace", "retrace", "td_multi", "gae_vtrace",
                   "trace", "prefix_sum") + tuple(
    e + sfx for sfx in NARROW
    for e in ("return", "td_lambda", "gae", "vtrace", "retrace", "trace", "prefix_sum"))


def per_estimator_roofline(torch, rlca, device, peak):
    """Each estimator alone at [4096, 1024] on its own workload's distributions."""
    return {est: time_workload(torch, rlca, device, peak, est,
                               workload_inputs(est, N_ENVS, SEQ_LEN, seed=100))
            for est in ESTIMATORS_1024}


# The workload configurations, each at its own shape and distributions.
CONFIGS = (
    ("gae_16x128", "gae", 16, 128),
    ("return_4096x128", "return", 4096, 128),
    ("td_lambda_0.9_4096x128", "td_lambda", 4096, 128),
    ("td_lambda_fused_0_0.9_1_4096x128", "td_multi", 4096, 128),
    ("gae_trunc_4096x1024", "gae", 4096, 1024),
    ("vtrace_8192x256", "vtrace", 8192, 256),
    ("retrace_2048x4096", "retrace", 2048, 4096),
)


def oracle_rows(est, ro, lo, hi):
    """The fp64 oracle, as it stands, for estimator `est` on rows [lo, hi)."""
    import oracle
    p = est_params(est, ro)
    sl = lambda a: None if a is None else a[lo:hi]
    fl = dict(terminated=sl(ro.terminated), truncated=sl(ro.truncated),
              trunc_value=sl(ro.trunc_value))
    if est == "return":
        oracle.discounted_return(sl(ro.reward), bootstrap=sl(ro.bootstrap), **fl,
                                 gamma=p["gamma"])
    elif est == "td_lambda":
        oracle.td_lambda(sl(ro.reward), sl(ro.value), bootstrap=sl(ro.bootstrap), **fl,
                         gamma=p["gamma"], lam=p["lam"])
    elif est == "td_multi":
        for lam in p["lams"]:
            oracle.td_lambda(sl(ro.reward), sl(ro.value), bootstrap=sl(ro.bootstrap), **fl,
                             gamma=p["gamma"], lam=lam)
    elif est == "gae":
        oracle.gae(sl(ro.reward), sl(ro.value), bootstrap=sl(ro.bootstrap), **fl,
                   gamma=p["gamma"], lam=p["lam"])
    elif est == "vtrace":
        oracle.vtrace(sl(ro.reward), sl(ro.value), sl(ro.log_rho), bootstrap=sl(ro.bootstrap),
                      **fl, gamma=p["gamma"], lam=p["lam"], rho_bar=p["rho_bar"],
                      c_bar=p["c_bar"], pg_rho_bar=p["pg_rho_bar"])
    else:
        oracle.retrace(sl(ro.reward), sl(ro.q_taken), sl(ro.expected_q), sl(ro.rho),
                       bootstrap_ev=sl(ro.bootstrap), **fl, gamma=p["gamma"], lam=p["lam"])


def oracle_rate(est, ro, seconds, pool=None, threads=1):
    """Timesteps/s of the oracle on the whole batch, repeated for about `seconds`: on one
    thread, or with rows split over `threads` threads of `pool`."""
    def run():
        if pool is None:
            oracle_rows(est, ro, 0, ro.N)
            return
        edges = np.linspace(0, ro.N, threads + 1).astype(int)
        futs = [pool.submit(oracle_rows, est, ro, a, b)
                for a, b in zip(edges[:-1], edges[1:]) if b > a]
        for f in futs:
            f.result()
    reps, t0 = 0, time.perf_counter()
    while True:
        run()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return round(reps * ro.N * ro.T / el, 1)


def per_config(torch, rlca, device, peak, cpu_seconds):
    """Every workload configuration timed alone at its own shape, with the fp64 oracle
    timed beside it on one host thread and on every host core."""
    import concurrent.futures
    import oracle
    oracle.build()
    threads = host_threads()
    out = {}
    with concurrent.futures.ThreadPoolExecutor(threads) as pool:
        for name, est, N, T in CONFIGS:
            ro = sr.gae_small(N=N, T=T, seed=100) if name == "gae_16x128" else \
                workload_inputs(est, N, T, seed=100)
            out[name] = time_workload(torch, rlca, device, peak, est, ro)
            if cpu_seconds > 0:
                out[name]["oracle_timesteps_per_s"] = {
                    "single_thread": oracle_rate(est, ro, cpu_seconds),
                    "all_cores": oracle_rate(est, ro, cpu_seconds, pool, threads),
                    "cores": threads}
    return out


def e2e_run(torch, rlca, ro, device, n_steps):
    """Public API end to end with the step's inputs and results in pinned host memory.

    Headline: the rollout tensors are pinned host memory and `rlca_gae` is called on them
    directly. On GB300 the kernel reads the inputs and writes advantages and returns in
    place over NVLink-C2C, so every byte crosses the link once, inside the timed call.
    For comparison, the same steps with explicit copies: double-buffered on three
    streams (step i+1's inputs copy in while step i runs and its results copy out), and
    one after another on one stream."""
    names = ("reward", "value", "terminated", "truncated", "trunc_value", "bootstrap")
    host = {k: torch.from_numpy(getattr(ro, k)).pin_memory() for k in names}
    res_h = (torch.empty((ro.N, ro.T), dtype=torch.float32).pin_memory(),
             torch.empty((ro.N, ro.T), dtype=torch.float32).pin_memory())
    params = ro.params
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = 2 * res_h[0].numel() * 4

    def call(src, adv, ret):
        rlca.rlca_gae(src["reward"], src["value"], src["terminated"], src["truncated"],
                      src["trunc_value"], src["bootstrap"], gamma=params["gamma"],
                      lam=params["lam"], advantages=adv, returns=ret)

    def timed(run_steps, streams=()):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream(device)
        e0.record(cur)
        for st in streams:
            st.wait_event(e0)
        run_steps()
        for st in streams:
            cur.wait_stream(st)
        e1.record(cur)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    # Zero-copy: one call per step on host tensors.
    for _ in range(3):
        call(host, *res_h)
    ms_zero = timed(lambda: [call(host, *res_h) for _ in range(n_steps)])
    torch.cuda.synchronize()
    dev = {k: v.to(device) for k, v in host.items()}
    ref = (torch.empty((ro.N, ro.T), device=device), torch.empty((ro.N, ro.T), device=device))
    call(dev, *ref)
    torch.cuda.synchronize()
    ok = bool(torch.equal(res_h[0], ref[0].cpu()) and torch.equal(res_h[1], ref[1].cpu()))

    # Explicit copies, double-buffered over three streams.
    devs = [{k: torch.empty_like(v, device=device) for k, v in host.items()} for _ in range(2)]
    outs = [(torch.empty((ro.N, ro.T), device=device), torch.empty((ro.N, ro.T), device=device))
            for _ in range(2)]
    s_in, s_run, s_out = (torch.cuda.Stream(device) for _ in range(3))
    ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]
    in_ready, run_done, out_done = ev(), ev(), ev()

    def step(i):
        b = i & 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(run_done[b])  # the call two steps back has read these inputs
            for k in names:
                devs[b][k].copy_(host[k], non_blocking=True)
            in_ready[b].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(in_ready[b])
            s_run.wait_event(out_done[b])  # results two steps back have been copied out
            call(devs[b], *outs[b])
            run_done[b].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(run_done[b])
            res_h[0].copy_(outs[b][0], non_blocking=True)
            res_h[1].copy_(outs[b][1], non_blocking=True)
            out_done[b].record(s_out)

    for i in range(4):
        step(i)
    ms_pipe = timed(lambda: [step(i) for i in range(n_steps)], (s_in, s_run, s_out))

    def serial():
        with torch.cuda.stream(s_run):
            for _ in range(n_steps):
                for k in names:
                    devs[0][k].copy_(host[k], non_blocking=True)
                call(devs[0], *outs[0])
                res_h[0].copy_(outs[0][0], non_blocking=True)
                res_h[1].copy_(outs[0][1], non_blocking=True)
    ms_serial = timed(serial, (s_run,))
    rate = lambda ms: round(ro.N * ro.T * n_steps / (ms * 1e-3), 1)
    return {"value": rate(ms_zero), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_steps,
            "ms_per_step": round(ms_zero / n_steps, 4),
            "mode": "zero-copy: rlca_gae called on pinned host tensors; the kernel reads "
                    "the inputs and writes the results in place over NVLink-C2C (the "
                    "byte counts are the host tensors' sizes; truncation values are "
                    "read only where a step is truncated)",
            "results_checked": ok,
            "copies_double_buffered": {"value": rate(ms_pipe),
                                       "ms_per_step": round(ms_pipe / n_steps, 4)},
            "copies_serial": {"value": rate(ms_serial),
                              "ms_per_step": round(ms_serial / n_steps, 4)}}


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def oracle_gae_rows(ro, lo, hi):
    """The fp64 oracle, as it stands, on rows [lo, hi) of the batch."""
    import oracle
    p = ro.params
    oracle.gae(ro.reward[lo:hi], ro.value[lo:hi], ro.terminated[lo:hi], ro.truncated[lo:hi],
               ro.trunc_value[lo:hi], ro.bootstrap[lo:hi], gamma=p["gamma"], lam=p["lam"])


def oracle_gae_all_cores(ro, rows, pool, threads):
    """The unchanged oracle on the first `rows` rows, split over `threads` host threads
    (the C call releases the interpreter lock, so the slices run in parallel)."""
    edges = np.linspace(0, rows, threads + 1).astype(int)
    futs = [pool.submit(oracle_gae_rows, ro, a, b)
            for a, b in zip(edges[:-1], edges[1:]) if b > a]
    for f in futs:
        f.result()


def cpu_baseline(ro, seconds):
    """The fp64 oracle as it stands on the full batch, repeated for about `seconds` of
    wall time: once on one thread, once split over every host core. The all-core figure
    is the reported value; the single-thread one rides along."""
    import concurrent.futures
    import oracle
    oracle.build()

    def timed(run):
        reps, t0 = 0, time.perf_counter()
        while True:
            run()
            reps += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return reps, el

    reps1, el1 = timed(lambda: oracle_gae_rows(ro, 0, ro.N))
    threads = host_threads()
    with concurrent.futures.ThreadPoolExecutor(threads) as pool:
        repsn, eln = timed(lambda: oracle_gae_all_cores(ro, ro.N, pool, threads))
    return {"value": round(repsn * ro.N * ro.T / eln, 1), "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "sample": f"full [{ro.N},{ro.T}] GAE batch (seed 0), {repsn} passes in "
                      f"{eln:.1f} s, rows split over {threads} threads, fp64 C reverse loop",
            "single_thread": {"value": round(reps1 * ro.N * ro.T / el1, 1), "cores": 1,
                              "sample": f"{reps1} passes in {el1:.1f} s"}}


def gpu_arm(args, rank, world, local_rank, dist):
    import torch

    import segmented_associative_scan_gb300 as rlca

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    rlca.lib()
    peak, peak_src = measured_peaks()

    # Distinct seeded batches, resident in HBM, rotating so their total exceeds L2.
    est = args.estimator
    N, T = args.num_envs, args.seq_len
    ro0 = workload_inputs(est, N, T, seed=1000 * rank)
    nbytes = algorithmic_bytes(est, ro0)
    n_sets = n_sets_for(nbytes)
    data_dtype = data_dtype_of(torch, est)
    sets = [DeviceSet(ro0, device, data_dtype)]
    for i in range(1, n_sets):
        sets.append(DeviceSet(workload_inputs(est, N, T, 1000 * rank + i), device, data_dtype))
    if args.workspace:
        for s in sets:
            s.ws = rlca.make_workspace(N, T, device)
    params = est_params(est, ro0)
    step_bytes = [algorithmic_bytes(est, s.ro) for s in sets]

    def step(i):
        launch(rlca, est, sets[i], params)

    K, W = args.steps, args.warmup
    for i in range(W):
        step(i % n_sets)
    torch.cuda.synchronize()
    G = n_sets * max(1, 96 // n_sets)
    graphs = [capture(torch, step, n_sets, G)] * (K // G)
    if K % G:
        graphs.append(capture(torch, step, n_sets, K % G))
    lead = graphs[0]  # untimed, keeps the GPU busy while the timed graphs are submitted
    lead.replay()
    torch.cuda.synchronize()
    kernel_bytes_per_step = sum(step_bytes[i % n_sets] for i in range(K)) / K

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    # Hold the GPU busy for ~0.5 s before timing so the clock samples see it under load.
    soak_end = time.time() + (0.0 if args.profile else 0.5)
    while time.time() < soak_end:
        lead.replay()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    ms = timed_replay(torch, graphs, lead)
    t1 = time.time()
    if dist is not None:
        dist.barrier()
    time.sleep(0.25)
    sampler.stop()
    clocks = sampler.summary(t0, t1)

    ms_max = max_over_ranks(ms, dist)
    if rank != 0:
        return None

    launch_us = 1000.0 * ms / K
    achieved = kernel_bytes_per_step / (launch_us * 1e-6) / 1e9
    value = job_throughput(world, N, T, K, ms_max)
    src_hash = kernel_source_hash()
    traffic = NCU_TRAFFIC.get((src_hash, est, N, T, bool(args.workspace)))
    in_name = est[len(base_est(est)) + 1:] if base_est(est) != est else "fp32"
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(ms_max / K, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic: seeded rollouts with the workload's distributions (no dataset)",
        "config": {
            "workload": WORKLOADS[est] if (N, T) == (N_ENVS, SEQ_LEN)
            else f"{est}, {in_name}, num_envs={N}, seq_len={T}", "estimator": est,
            "num_envs": N, "seq_len": T, "gamma": params["gamma"], "lambda": params.get("lam"),
            "input_sets": n_sets,
            "entry": "_ex entry point with a caller workspace" if args.workspace
                     else "plain entry point",
            "l2": (f"inputs larger than L2: {n_sets} distinct batches of "
                   f"{nbytes / 1e6:.1f} MB rotate ({n_sets * nbytes / 1e6:.0f} MB > "
                   f"{L2_BYTES / 1e6:.0f} MB L2)") if n_sets * nbytes > L2_BYTES else
                  (f"{n_sets} batches of {nbytes / 1e6:.2f} MB rotate; they fit in L2"),
            "timing": f"CUDA graphs of {min(G, K)} launches replayed between CUDA events on "
                      "the launch stream, after an untimed graph that keeps the GPU busy "
                      "while they are submitted; one fused kernel launch per step",
            "parallelism": f"replicas{world}: each GPU its own batch, no collective"},
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "traffic_kind": "ncu, one launch: dram__bytes_read.sum + 32 x "
                            "lts__t_sectors_srcunit_tex_op_write.sum (bytes the SMs wrote into "
                            "L2: the outputs stay in L2 until after a captured launch ends)",
            "kernel": kernel_desc(est, N, T, args.workspace,
                                  torch.cuda.get_device_properties(device).multi_processor_count),
            "algorithmic_bytes_per_launch": round(kernel_bytes_per_step),
            "launch_us": round(launch_us, 3), "peak_source": peak_src,
            "frac_of_8tbs": round(achieved / 8000.0, 4), "kernel_source": src_hash},
        "gpu_launches": K,
        "clocks": clocks,
    }
    if not args.no_e2e and est == "gae":
        result["e2e"] = e2e_run(torch, rlca, ro0, device, min(K, args.e2e_steps))
    del graphs, sets, lead
    torch.cuda.empty_cache()
    if world == 1 and args.cpu_seconds > 0 and est == "gae":
        result["cpu_baseline"] = cpu_baseline(ro0, args.cpu_seconds)
    if world == 1 and not args.no_estimators and (N, T) == (N_ENVS, SEQ_LEN):
        configs = per_config(torch, rlca, device, peak, min(1.0, args.cpu_seconds / 10.0))
        estimators = per_estimator_roofline(torch, rlca, device, peak)
        steady = configs.get(f"{est}_trunc_{N}x{T}") if est == "gae" else None
        if steady is not None:
            # The same kernel timed over ~300 back-to-back launches on other batches.
            result["roofline"]["launch_us_steady"] = steady["us_per_launch"]
            result["roofline"]["frac_steady"] = steady["frac"]
        if args.detail:
            with open(args.detail, "w") as f:
                json.dump({"configs": configs, "estimators": estimators}, f, indent=1)
        keep = ("us_per_launch", "frac", "ceiling_us", "frac_of_ceiling", "ncu_traffic_ratio",
                "inputs_exceed_l2", "oracle_timesteps_per_s")
        result["configs"] = {k: {f: v[f] for f in keep if f in v} for k, v in configs.items()}
        # Last key: each estimator alone at [4096, 1024], us per launch, fraction of the
        # measured peak and of its plain-copy ceiling.
        result["estimators"] = {
            k: [v["us_per_launch"], v["frac"]] + ([v["frac_of_ceiling"]]
                                                 if "frac_of_ceiling" in v else [])
            for k, v in estimators.items()}
    return result


# --------------------------------------------------------------------- reference arm

def reference_arm(args):
    """The fp64 CPU oracle as it stands, on every host core (rows split over threads),
    each step a bounded sample (the first rows) of the same [4096, 1024] GAE workload."""
    import concurrent.futures
    import oracle
    oracle.build()
    ro = workload_inputs("gae", N_ENVS, SEQ_LEN, seed=0)
    threads = host_threads()
    pool = concurrent.futures.ThreadPoolExecutor(threads)

    def run(rows):
        oracle_gae_all_cores(ro, rows, pool, threads)

    t0 = time.perf_counter()
    run(min(N_ENVS, 64 * threads))
    per_row = (time.perf_counter() - t0) / min(N_ENVS, 64 * threads)
    budget = args.reference_seconds / max(1, args.steps + args.warmup)
    rows = int(max(threads, min(N_ENVS, budget / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        run(rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run(rows)
    el = time.perf_counter() - t0
    pool.shutdown()
    value = rows * SEQ_LEN * args.steps / el
    sample = (f"first {rows} of {N_ENVS} envs x {SEQ_LEN} steps per step, rows split "
              f"over {threads} threads, fp64 C reverse loop")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * el / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded rollouts with the workload's distributions (no dataset)",
        "config": {"workload": WORKLOAD, "estimator": "gae", "num_envs": N_ENVS,
                   "seq_len": SEQ_LEN, "sample_envs": rows},
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("rlca", "reference"), default="rlca")
    ap.add_argument("--num-envs", type=int, default=N_ENVS)
    ap.add_argument("--seq-len", type=int, default=SEQ_LEN)
    ap.add_argument("--estimator", choices=tuple(WORKLOADS), default="gae",
                    help="estimator timed in the main loop (the metric's workload is gae)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=60.0)
    ap.add_argument("--workspace", action="store_true",
                    help="give every call a look-back workspace (the _ex entry points of the "
                         "five reverse estimators)")
    ap.add_argument("--detail", default=None,
                    help="also write the full per-configuration and per-estimator tables "
                         "to this JSON file")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-estimators", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="short run for profilers: no clock soak, e2e, per-estimator table "
                         "or CPU baseline")
    args = ap.parse_args()
    if args.profile:
        args.no_e2e = args.no_estimators = True
        args.cpu_seconds = 0.0
    if args.steps < 1 or args.warmup < 0:
        ap.error("--steps must be >= 1 and --warmup >= 0")
    if args.workspace and args.estimator not in ("gae", "return", "td_lambda", "vtrace",
                                                 "retrace"):
        ap.error("--workspace applies to the five fp32 reverse estimators")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args)), flush=True)
        return

    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        dist = tdist
    try:
        res = gpu_arm(args, rank, world, local_rank, dist)
    finally:
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
