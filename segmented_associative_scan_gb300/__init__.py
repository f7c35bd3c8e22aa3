"""Python binding of librlca: RL credit assignment as fused segmented reverse affine
scans on one GB300 (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA kernels of
``librlca.so``; PyTorch supplies device memory and the current stream. There is no CPU
fallback: if the library is not built, every call raises.

The functions carry the names of the C entry points (``include/rlca.h``) and take
torch tensors:
  - per-step tensors: 2-D [N, T], unit stride along T, all with the same row stride;
    float32 data (or all bfloat16 / all float16, which select the _bf16 / _fp16 entry
    points), uint8 or bool flags;
  - per-env bootstrap values: float32 [N] (optional);
  - every tensor is on one CUDA device or in pinned host memory (read and written in
    place by the kernels over NVLink-C2C);
  - outputs are allocated (same row stride as the inputs; pinned host memory when the
    reward tensor is there) unless passed in.
Work is enqueued on ``torch.cuda.current_stream()``; nothing synchronises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librlca.so")

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
SIGNATURES = {
    "rlca_version": ([], ctypes.c_int),
    "rlca_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "rlca_discounted_return": ([_P, _P, _P, _P, _P, _F, _I64, _I64, _I64, _P, _P],
                               ctypes.c_int),
    "rlca_td_lambda": ([_P, _P, _P, _P, _P, _P, _F, _F, _I64, _I64, _I64, _P, _P],
                       ctypes.c_int),
    "rlca_gae": ([_P, _P, _P, _P, _P, _P, _F, _F, _I64, _I64, _I64, _P, _P, _P],
                 ctypes.c_int),
    "rlca_vtrace": ([_P, _P, _P, _P, _P, _P, _P, _F, _F, _F, _F, _F, _I64, _I64, _I64, _P,
                     _P, _P], ctypes.c_int),
    "rlca_retrace": ([_P, _P, _P, _P, _P, _P, _P, _P, _F, _F, _I64, _I64, _I64, _P, _P],
                     ctypes.c_int),
    "rlca_td_lambda_multi": ([_P, _P, _P, _P, _P, _P, _F, _P, ctypes.c_int, _I64, _I64, _I64,
                              _P, _P], ctypes.c_int),
    "rlca_gae_vtrace": ([_P, _P, _P, _P, _P, _P, _P, _F, _F, _F, _F, _F, _F, _I64, _I64, _I64,
                         _P, _P, _P, _P, _P], ctypes.c_int),
    "rlca_eligibility_trace": ([_P, _P, _P, _P, _F, _I64, _I64, _I64, _P, _P], ctypes.c_int),
    "rlca_episodic_prefix_sum": ([_P, _P, _P, _P, _I64, _I64, _I64, _P, _P], ctypes.c_int),
    "rlca_workspace_bytes": ([_I64, _I64], ctypes.c_size_t),
    "rlca_workspace_check": ([_P, _P], ctypes.c_int),
    "rlca_testing_lookback_stall": ([_P, _P, _I64, _I64, _P, _P, ctypes.c_size_t, ctypes.c_int,
                                     _P], ctypes.c_int),
}
SIGNATURES["rlca_gae_noalloc"] = SIGNATURES["rlca_gae"]
# Measurement only (include/rlca_measure.h).
SIGNATURES["rlca_measure_copy"] = ([_P, ctypes.c_int, ctypes.c_int, _P, ctypes.c_int, _P,
                                    ctypes.c_int, _I64, ctypes.c_int, _P], ctypes.c_int)
# 16-bit-input variants: the same argument list (the data pointers hold bf16 or fp16).
for _name in ("rlca_discounted_return", "rlca_td_lambda", "rlca_gae", "rlca_vtrace",
              "rlca_retrace", "rlca_eligibility_trace", "rlca_episodic_prefix_sum"):
    SIGNATURES[_name + "_bf16"] = SIGNATURES[_name]
    SIGNATURES[_name + "_fp16"] = SIGNATURES[_name]
# The _ex variants take (workspace, workspace_bytes) before the stream.
for _name in ("rlca_discounted_return", "rlca_td_lambda", "rlca_gae", "rlca_vtrace",
              "rlca_retrace"):
    _args, _res = SIGNATURES[_name]
    SIGNATURES[_name + "_ex"] = (_args[:-1] + [_P, ctypes.c_size_t, _P], _res)

_lib = None


def build(force: bool = False) -> str:
    """Compile librlca.so in-tree (nvcc, sm_103a)."""
    from . import buildlib as _build
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded C library with argument types set. Raises if it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "segmented_associative_scan_gb300.build()")
        cdll = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(cdll, name)
            fn.argtypes = args
            fn.restype = res
        _lib = cdll
    return _lib


class RlcaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {lib().rlca_status_string(status).decode()} (status {status})")


def _check(fn: str, status: int):
    if status != 0:
        raise RlcaError(fn, status)


class _Rows:
    """Shape/stride bookkeeping shared by the per-step tensors of one call.

    Tensors live on one CUDA device, or in pinned host memory, which the kernels read
    and write in place (mixing the two is allowed). A call whose first per-step tensor
    is in pinned host memory runs on the current CUDA device and allocates missing
    outputs in pinned host memory."""

    def __init__(self, ref: torch.Tensor):
        if ref.dim() != 2:
            raise ValueError("per-step tensors must be 2-D [num_envs, seq_len]")
        self.N, self.T = ref.shape
        self.ld = ref.stride(0) if self.N > 1 else max(ref.stride(0), self.T)
        self.host = not ref.is_cuda
        if self.host and not ref.is_pinned():
            raise ValueError("host tensors must be in pinned memory (pin_memory())")
        self.device = (torch.device("cuda", torch.cuda.current_device()) if self.host
                       else ref.device)

    def _reachable(self, t, name):
        if t.is_cuda:
            if t.device != self.device:
                raise ValueError(f"{name} must be on {self.device} or in pinned host memory")
        elif not t.is_pinned():
            raise ValueError(f"{name} must be on {self.device} or in pinned host memory")

    def ptr(self, t, name, dtypes, optional=False):
        if t is None:
            if optional:
                return None
            raise ValueError(f"{name} is required")
        self._reachable(t, name)
        if t.dtype not in dtypes:
            raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
        if tuple(t.shape) != (self.N, self.T):
            raise ValueError(f"{name}: shape {tuple(t.shape)} != {(self.N, self.T)}")
        if self.T > 1 and t.stride(1) != 1:
            raise ValueError(f"{name}: steps must be contiguous (stride(1) == 1)")
        if self.N > 1 and t.stride(0) != self.ld:
            raise ValueError(f"{name}: row stride {t.stride(0)} != {self.ld}")
        return t.data_ptr() or None

    def vec_ptr(self, t, name):
        if t is None:
            return None
        self._reachable(t, name)
        if t.dtype != torch.float32 or t.dim() != 1 or t.shape[0] != self.N:
            raise ValueError(f"{name} must be a float32 [{self.N}] tensor")
        if self.N > 1 and t.stride(0) != 1:
            raise ValueError(f"{name} must be contiguous")
        return t.data_ptr() or None

    def out(self, t, name):
        if t is None:
            shape = (self.N, max(self.ld, self.T))
            buf = (torch.empty(shape, dtype=torch.float32, pin_memory=True) if self.host
                   else torch.empty(shape, dtype=torch.float32, device=self.device))
            t = buf[:, :self.T]
        self.ptr(t, name, (torch.float32,))
        return t


_F32 = (torch.float32,)
_FLAG = (torch.uint8, torch.bool)


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def workspace_bytes(N: int, T: int) -> int:
    """Bytes of look-back workspace an [N, T] call needs (0: none needed)."""
    return int(lib().rlca_workspace_bytes(N, T))


def make_workspace(N: int, T: int, device="cuda") -> torch.Tensor | None:
    """A zero-filled workspace tensor for the _ex (look-back) path, or None when
    T fits one tile. PyTorch allocates it; the library never allocates."""
    n = workspace_bytes(N, T)
    return torch.zeros(n, dtype=torch.uint8, device=device) if n else None


def workspace_check(workspace: torch.Tensor) -> int:
    """Synchronise the current stream and return the workspace's status
    (0, or -7 after a look-back wait gave up; the record is then cleared)."""
    return int(lib().rlca_workspace_check(workspace.data_ptr(), _stream(workspace.device)))


def _narrow(dd):
    """The 16-bit data dtype of an allowed-dtype tuple, or None for fp32."""
    return dd[0] if dd[0] in _NARROW else None


# Entry-point suffix of each 16-bit data dtype.
_NARROW = {torch.bfloat16: "_bf16", torch.float16: "_fp16"}


def _data_dtype(t):
    """Per-step data inputs are all fp32, all bf16 or all fp16; returns the allowed dtype
    tuple (the first per-step tensor decides)."""
    if t.dtype in _NARROW:
        return (t.dtype,)
    return _F32


def _call(name, args, workspace, stream, narrow=None):
    """Call the plain entry point, its _bf16 / _fp16 variant for 16-bit inputs (`narrow`,
    the data dtype), or its _ex variant when a workspace is given."""
    if narrow is not None:
        if workspace is not None:
            raise ValueError("the 16-bit input entry points take no workspace")
        return getattr(lib(), name + _NARROW[narrow])(*args, stream)
    if workspace is None:
        return getattr(lib(), name)(*args, stream)
    if not workspace.is_cuda or workspace.dtype != torch.uint8:
        raise ValueError("workspace must be a CUDA uint8 tensor")
    return getattr(lib(), name + "_ex")(*args, workspace.data_ptr(),
                                        workspace.numel(), stream)


def rlca_discounted_return(reward, terminated, truncated=None, trunc_value=None,
                           bootstrap=None, gamma=0.99, returns=None, workspace=None):
    g = _Rows(reward)
    dd = _data_dtype(reward)
    args = (g.ptr(reward, "reward", dd), g.ptr(terminated, "terminated", _FLAG),
            g.ptr(truncated, "truncated", _FLAG, True),
            g.ptr(trunc_value, "trunc_value", dd, truncated is None),
            g.vec_ptr(bootstrap, "bootstrap"))
    returns = g.out(returns, "returns")
    _check("rlca_discounted_return", _call(
        "rlca_discounted_return", (*args, gamma, g.N, g.T, g.ld, returns.data_ptr() or None),
        workspace, _stream(g.device), _narrow(dd)))
    return returns


def rlca_td_lambda(reward, value, terminated, truncated=None, trunc_value=None,
                   bootstrap=None, gamma=0.99, lam=0.95, targets=None, workspace=None):
    g = _Rows(reward)
    dd = _data_dtype(reward)
    args = (g.ptr(reward, "reward", dd), g.ptr(value, "value", dd),
            g.ptr(terminated, "terminated", _FLAG), g.ptr(truncated, "truncated", _FLAG, True),
            g.ptr(trunc_value, "trunc_value", dd, truncated is None),
            g.vec_ptr(bootstrap, "bootstrap"))
    targets = g.out(targets, "targets")
    _check("rlca_td_lambda", _call(
        "rlca_td_lambda", (*args, gamma, lam, g.N, g.T, g.ld, targets.data_ptr() or None),
        workspace, _stream(g.device), _narrow(dd)))
    return targets


def rlca_gae(reward, value, terminated, truncated=None, trunc_value=None, bootstrap=None,
             gamma=0.99, lam=0.95, advantages=None, returns=None, want_returns=True,
             workspace=None):
    g = _Rows(reward)
    dd = _data_dtype(reward)
    args = (g.ptr(reward, "reward", dd), g.ptr(value, "value", dd),
            g.ptr(terminated, "terminated", _FLAG), g.ptr(truncated, "truncated", _FLAG, True),
            g.ptr(trunc_value, "trunc_value", dd, truncated is None),
            g.vec_ptr(bootstrap, "bootstrap"))
    advantages = g.out(advantages, "advantages")
    returns = g.out(returns, "returns") if (want_returns or returns is not None) else None
    _check("rlca_gae", _call(
        "rlca_gae", (*args, gamma, lam, g.N, g.T, g.ld, advantages.data_ptr() or None,
                     returns.data_ptr() or None if returns is not None else None),
        workspace, _stream(g.device), _narrow(dd)))
    return advantages, returns


def rlca_vtrace(reward, value, log_rho, terminated, truncated=None, trunc_value=None,
                bootstrap=None, gamma=0.99, lam=1.0, rho_bar=1.0, c_bar=1.0,
                pg_rho_bar=None, vs=None, pg_advantages=None, want_pg=True, workspace=None):
    g = _Rows(reward)
    dd = _data_dtype(reward)
    args = (g.ptr(reward, "reward", dd), g.ptr(value, "value", dd),
            g.ptr(log_rho, "log_rho", dd), g.ptr(terminated, "terminated", _FLAG),
            g.ptr(truncated, "truncated", _FLAG, True),
            g.ptr(trunc_value, "trunc_value", dd, truncated is None),
            g.vec_ptr(bootstrap, "bootstrap"))
    vs = g.out(vs, "vs")
    pg = g.out(pg_advantages, "pg_advantages") if (want_pg or pg_advantages is not None) \
        else None
    if pg_rho_bar is None:
        pg_rho_bar = rho_bar
    _check("rlca_vtrace", _call(
        "rlca_vtrace", (*args, gamma, lam, rho_bar, c_bar, pg_rho_bar, g.N, g.T, g.ld,
                        vs.data_ptr() or None,
                        pg.data_ptr() or None if pg is not None else None),
        workspace, _stream(g.device), _narrow(dd)))
    return vs, pg


def rlca_gae_vtrace(reward, value, log_rho, terminated, truncated=None, trunc_value=None,
                    bootstrap=None, gamma=0.99, lam=0.95, lam_vtrace=1.0, rho_bar=1.0,
                    c_bar=1.0, pg_rho_bar=None, advantages=None, returns=None, vs=None,
                    pg_advantages=None, want_returns=True, want_pg=True):
    """GAE and V-trace from one read of the inputs (fp32): returns (advantages, returns,
    vs, pg_advantages); returns / pg_advantages are None when not wanted."""
    g = _Rows(reward)
    args = (g.ptr(reward, "reward", _F32), g.ptr(value, "value", _F32),
            g.ptr(log_rho, "log_rho", _F32), g.ptr(terminated, "terminated", _FLAG),
            g.ptr(truncated, "truncated", _FLAG, True),
            g.ptr(trunc_value, "trunc_value", _F32, truncated is None),
            g.vec_ptr(bootstrap, "bootstrap"))
    adv = g.out(advantages, "advantages")
    ret = g.out(returns, "returns") if (want_returns or returns is not None) else None
    vs = g.out(vs, "vs")
    pg = g.out(pg_advantages, "pg_advantages") if (want_pg or pg_advantages is not None) \
        else None
    if pg_rho_bar is None:
        pg_rho_bar = rho_bar
    ptr = lambda t: None if t is None else (t.data_ptr() or None)
    _check("rlca_gae_vtrace", lib().rlca_gae_vtrace(
        *args, gamma, lam, lam_vtrace, rho_bar, c_bar, pg_rho_bar, g.N, g.T, g.ld, ptr(adv),
        ptr(ret), ptr(vs), ptr(pg), _stream(g.device)))
    return adv, ret, vs, pg


def rlca_retrace(reward, q_taken, expected_q, rho, terminated, truncated=None,
                 trunc_value=None, bootstrap_ev=None, gamma=0.99, lam=0.95, q_ret=None,
                 workspace=None):
    g = _Rows(reward)
    dd = _data_dtype(reward)
    args = (g.ptr(reward, "reward", dd), g.ptr(q_taken, "q_taken", dd),
            g.ptr(expected_q, "expected_q", dd), g.ptr(rho, "rho", dd),
            g.ptr(terminated, "terminated", _FLAG), g.ptr(truncated, "truncated", _FLAG, True),
            g.ptr(trunc_value, "trunc_value", dd, truncated is None),
            g.vec_ptr(bootstrap_ev, "bootstrap_ev"))
    q_ret = g.out(q_ret, "q_ret")
    _check("rlca_retrace", _call(
        "rlca_retrace", (*args, gamma, lam, g.N, g.T, g.ld, q_ret.data_ptr() or None),
        workspace, _stream(g.device), _narrow(dd)))
    return q_ret


def rlca_td_lambda_multi(reward, value, terminated, truncated=None, trunc_value=None,
                         bootstrap=None, gamma=0.99, lams=(0.0, 0.9, 1.0), targets=None):
    """TD(lambda) targets for several lambdas (at most 4) from one read of the inputs.
    Returns a list of [N, T] tensors, one per lambda."""
    g = _Rows(reward)
    args = (g.ptr(reward, "reward", _F32), g.ptr(value, "value", _F32),
            g.ptr(terminated, "terminated", _FLAG), g.ptr(truncated, "truncated", _FLAG, True),
            g.ptr(trunc_value, "trunc_value", _F32, truncated is None),
            g.vec_ptr(bootstrap, "bootstrap"))
    lams = [float(x) for x in lams]
    if targets is None:
        targets = [None] * len(lams)
    targets = [g.out(t, f"targets[{k}]") for k, t in enumerate(targets)]
    lam_arr = (ctypes.c_float * len(lams))(*lams)
    out_arr = (ctypes.c_void_p * len(lams))(*[t.data_ptr() or None for t in targets])
    _check("rlca_td_lambda_multi", lib().rlca_td_lambda_multi(
        *args, gamma, lam_arr, len(lams), g.N, g.T, g.ld, out_arr, _stream(g.device)))
    return targets


def rlca_eligibility_trace(x, terminated, truncated=None, init=None, decay=0.95,
                           traces=None):
    """Forward accumulating trace e_t = x_t + decay e_{t-1}, fresh after an episode ends,
    e_{-1} = init."""
    g = _Rows(x)
    dd = _data_dtype(x)
    args = (g.ptr(x, "x", dd), g.ptr(terminated, "terminated", _FLAG),
            g.ptr(truncated, "truncated", _FLAG, True), g.vec_ptr(init, "init"))
    traces = g.out(traces, "traces")
    _check("rlca_eligibility_trace", _call(
        "rlca_eligibility_trace", (*args, decay, g.N, g.T, g.ld, traces.data_ptr() or None),
        None, _stream(g.device), _narrow(dd)))
    return traces


def rlca_episodic_prefix_sum(x, terminated, truncated=None, init=None, sums=None):
    """Forward sum of x within each episode, S_{-1} = init."""
    g = _Rows(x)
    dd = _data_dtype(x)
    args = (g.ptr(x, "x", dd), g.ptr(terminated, "terminated", _FLAG),
            g.ptr(truncated, "truncated", _FLAG, True), g.vec_ptr(init, "init"))
    sums = g.out(sums, "sums")
    _check("rlca_episodic_prefix_sum", _call(
        "rlca_episodic_prefix_sum", (*args, g.N, g.T, g.ld, sums.data_ptr() or None),
        None, _stream(g.device), _narrow(dd)))
    return sums


def measure_copy(inputs, flags, outputs, chunks=1):
    """Measurement only (rlca_measure_copy): one launch that reads every element of the
    `inputs` (all float32, or all bfloat16 / float16) and uint8/bool `flags` and writes
    every element of the fp32 `outputs`, in the estimator kernels' launch shape (`chunks`
    256-element chunks per warp). All tensors are contiguous, on one CUDA device, with
    the same number of elements."""
    n = inputs[0].numel()
    dev = inputs[0].device
    in_dt = _data_dtype(inputs[0])
    for t, dts in [(t, in_dt) for t in inputs] + [(t, _F32) for t in outputs] + \
            [(t, _FLAG) for t in flags]:
        if not t.is_cuda or t.device != dev or not t.is_contiguous() or t.numel() != n:
            raise ValueError("measure_copy: contiguous tensors of one size on one device")
        if t.dtype not in dts:
            raise TypeError(f"measure_copy: dtype {t.dtype} not in {dts}")
    arr = lambda ts: (ctypes.c_void_p * max(1, len(ts)))(*[t.data_ptr() for t in ts])
    _check("rlca_measure_copy", lib().rlca_measure_copy(
        arr(inputs), len(inputs), inputs[0].element_size(), arr(flags), len(flags),
        arr(outputs), len(outputs), n, chunks, _stream(dev)))


# Short names.
discounted_return = rlca_discounted_return
td_lambda = rlca_td_lambda
gae = rlca_gae
vtrace = rlca_vtrace
gae_vtrace = rlca_gae_vtrace
retrace = rlca_retrace
td_lambda_multi = rlca_td_lambda_multi
eligibility_trace = rlca_eligibility_trace
episodic_prefix_sum = rlca_episodic_prefix_sum
