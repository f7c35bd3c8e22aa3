"""fp64 CPU oracle for RL credit assignment (plain reverse loops in C).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU baseline
call it. The product path never imports this package, and this package never imports
the product package; they share only the seeded input generators.

Each function follows the textbook recursion of one estimator, with the boundary rules
of "rl-triton: High-Performance Triton GPU Kernels for Reinforcement Learning Credit
Assignment", Method section 3 (termination: successor value 0; truncation: supplied
bootstrap value; window end t = T-1: per-env bootstrap, counted once). The formulas are
spelled out in ``rlca_oracle.c``.

Also the forward-time scans: eligibility traces and episodic prefix sums.

Parity pins (tests/test_oracle_pins.py, tests/test_oracle_forward_pins.py): closed-form
returns and traces, hand-computed golden
examples, GAE(lambda=1) = return - V, GAE(lambda=0) = TD error, TD(lambda) = GAE returns,
non-recursive sum definitions (GAE, lambda-return as weighted n-step returns, IMPALA
V-trace sum, Retrace sum), on-policy reductions of V-trace and Retrace, and per-episode
recomputation (no leakage across episode boundaries).

Inputs are numpy arrays: float32 [N, ld] data (first T columns used), uint8 [N, ld]
flags, float32 [N] bootstrap. Scalars (gamma, lambda, clips) are rounded to float32 and
widened, so the oracle sees exactly the parameter values the fp32 kernels see.
Outputs are float64 [N, T].
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rlca_oracle.c")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, portable flags only)."""
    if force or not os.path.exists(_OUT) or os.path.getmtime(_OUT) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_OUT), exist_ok=True)
        tmp = _OUT + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _OUT)
    return _OUT


_F = ctypes.c_void_p
_I = ctypes.c_int64
_D = ctypes.c_double
_SIGS = {
    "oracle_discounted_return": [_F, _F, _F, _F, _F, _D, _I, _I, _I, _F],
    "oracle_gae": [_F, _F, _F, _F, _F, _F, _D, _D, _I, _I, _I, _F, _F],
    "oracle_td_lambda": [_F, _F, _F, _F, _F, _F, _D, _D, _I, _I, _I, _F],
    "oracle_vtrace": [_F, _F, _F, _F, _F, _F, _F, _D, _D, _D, _D, _D, _I, _I, _I, _F, _F],
    "oracle_retrace": [_F, _F, _F, _F, _F, _F, _F, _F, _D, _D, _I, _I, _I, _F],
    "oracle_eligibility_trace": [_F, _F, _F, _F, _D, _I, _I, _I, _F],
    "oracle_episodic_prefix_sum": [_F, _F, _F, _F, _I, _I, _I, _F],
}


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        for name, args in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = None
        _lib = lib
    return _lib


def _p(a, dtype):
    if a is None:
        return None, None
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def _f32(x) -> float:
    return float(np.float32(x))


def _shape(reward, T):
    N, ld = reward.shape
    T = ld if T is None else int(T)
    assert 0 <= T <= ld
    return N, T, ld


def _common(reward, terminated, truncated, trunc_value, bootstrap):
    keep = []
    ptrs = []
    for a, dt in ((reward, np.float32), (terminated, np.uint8), (truncated, np.uint8),
                  (trunc_value, np.float32), (bootstrap, np.float32)):
        arr, ptr = _p(a, dt)
        keep.append(arr)
        ptrs.append(ptr)
    if truncated is not None:
        assert trunc_value is not None, "trunc_value is required with truncated"
    return keep, ptrs


def discounted_return(reward, terminated, truncated=None, trunc_value=None, bootstrap=None,
                      gamma=0.99, T=None):
    N, T, ld = _shape(reward, T)
    keep, (r, d, tr, tv, b) = _common(reward, terminated, truncated, trunc_value, bootstrap)
    out = np.empty((N, T), np.float64)
    _load().oracle_discounted_return(r, d, tr, tv, b, _f32(gamma), N, T, ld, out.ctypes.data)
    return out


def gae(reward, value, terminated, truncated=None, trunc_value=None, bootstrap=None,
        gamma=0.99, lam=0.95, T=None):
    N, T, ld = _shape(reward, T)
    keep, (r, d, tr, tv, b) = _common(reward, terminated, truncated, trunc_value, bootstrap)
    v_arr, v = _p(value, np.float32)
    adv = np.empty((N, T), np.float64)
    ret = np.empty((N, T), np.float64)
    _load().oracle_gae(r, v, d, tr, tv, b, _f32(gamma), _f32(lam), N, T, ld,
                       adv.ctypes.data, ret.ctypes.data)
    return adv, ret


def td_lambda(reward, value, terminated, truncated=None, trunc_value=None, bootstrap=None,
              gamma=0.99, lam=0.95, T=None):
    N, T, ld = _shape(reward, T)
    keep, (r, d, tr, tv, b) = _common(reward, terminated, truncated, trunc_value, bootstrap)
    v_arr, v = _p(value, np.float32)
    out = np.empty((N, T), np.float64)
    _load().oracle_td_lambda(r, v, d, tr, tv, b, _f32(gamma), _f32(lam), N, T, ld,
                             out.ctypes.data)
    return out


def vtrace(reward, value, log_rho, terminated, truncated=None, trunc_value=None,
           bootstrap=None, gamma=0.99, lam=1.0, rho_bar=1.0, c_bar=1.0, pg_rho_bar=None,
           T=None):
    N, T, ld = _shape(reward, T)
    keep, (r, d, tr, tv, b) = _common(reward, terminated, truncated, trunc_value, bootstrap)
    v_arr, v = _p(value, np.float32)
    l_arr, lr = _p(log_rho, np.float32)
    if pg_rho_bar is None:
        pg_rho_bar = rho_bar
    vs = np.empty((N, T), np.float64)
    pg = np.empty((N, T), np.float64)
    _load().oracle_vtrace(r, v, lr, d, tr, tv, b, _f32(gamma), _f32(lam), _f32(rho_bar),
                          _f32(c_bar), _f32(pg_rho_bar), N, T, ld, vs.ctypes.data,
                          pg.ctypes.data)
    return vs, pg


def retrace(reward, q_taken, expected_q, rho, terminated, truncated=None, trunc_value=None,
            bootstrap_ev=None, gamma=0.99, lam=0.95, T=None):
    N, T, ld = _shape(reward, T)
    keep, (r, d, tr, tv, b) = _common(reward, terminated, truncated, trunc_value,
                                      bootstrap_ev)
    q_arr, q = _p(q_taken, np.float32)
    e_arr, e = _p(expected_q, np.float32)
    p_arr, p = _p(rho, np.float32)
    out = np.empty((N, T), np.float64)
    _load().oracle_retrace(r, q, e, p, d, tr, tv, b, _f32(gamma), _f32(lam), N, T, ld,
                           out.ctypes.data)
    return out


def _forward_args(x, terminated, truncated, init):
    keep = []
    ptrs = []
    for a, dt in ((x, np.float32), (terminated, np.uint8), (truncated, np.uint8),
                  (init, np.float32)):
        arr, ptr = _p(a, dt)
        keep.append(arr)
        ptrs.append(ptr)
    return keep, ptrs


def eligibility_trace(x, terminated, truncated=None, init=None, decay=0.95, T=None):
    """Forward accumulating trace e_t = x_t + decay * e_{t-1}, fresh after an episode end,
    e_{-1} = init (rl-triton technical summary, Method section 1: the forward-time mirror
    of the recurrence)."""
    N, T, ld = _shape(x, T)
    keep, (xp, d, tr, ini) = _forward_args(x, terminated, truncated, init)
    out = np.empty((N, T), np.float64)
    _load().oracle_eligibility_trace(xp, d, tr, ini, _f32(decay), N, T, ld, out.ctypes.data)
    return out


def episodic_prefix_sum(x, terminated, truncated=None, init=None, T=None):
    """Forward sum within each episode (Method section 1: episodic prefix sums)."""
    N, T, ld = _shape(x, T)
    keep, (xp, d, tr, ini) = _forward_args(x, terminated, truncated, init)
    out = np.empty((N, T), np.float64)
    _load().oracle_episodic_prefix_sum(xp, d, tr, ini, N, T, ld, out.ctypes.data)
    return out
