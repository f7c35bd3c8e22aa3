"""Shared helpers of the GPU parity tests: run one estimator on the CUDA path (through
the C-ABI binding) and on the fp64 oracle, from the same seeded host arrays, and
compare with the tolerance max|gpu - oracle| <= 1e-4 * (1 + max|oracle|)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import segmented_associative_scan_gb300 as rlca

ESTIMATORS = ("return", "td_lambda", "gae", "vtrace", "retrace")
TOL = 1e-4
GUARD = 64           # sentinel elements before and after every buffer
SENTINEL = -7777.25  # written around every output; must survive every call

DEFAULT_PARAMS = {
    "return": dict(gamma=0.99),
    "td_lambda": dict(gamma=0.99, lam=0.9),
    "gae": dict(gamma=0.99, lam=0.95),
    "vtrace": dict(gamma=0.99, lam=1.0, rho_bar=1.0, c_bar=1.0, pg_rho_bar=1.0),
    "retrace": dict(gamma=0.99, lam=0.95),
}

OUTPUTS = {
    "return": ("returns",), "td_lambda": ("targets",), "gae": ("advantages", "returns"),
    "vtrace": ("vs", "pg_advantages"), "retrace": ("q_ret",),
}


def run_oracle(est, ro, params):
    p = dict(DEFAULT_PARAMS[est], **params)
    fl = dict(terminated=ro.terminated, truncated=ro.truncated, trunc_value=ro.trunc_value)
    if est == "return":
        return {"returns": oracle.discounted_return(ro.reward, bootstrap=ro.bootstrap, **fl,
                                                    gamma=p["gamma"])}
    if est == "td_lambda":
        return {"targets": oracle.td_lambda(ro.reward, ro.value, bootstrap=ro.bootstrap, **fl,
                                            gamma=p["gamma"], lam=p["lam"])}
    if est == "gae":
        adv, ret = oracle.gae(ro.reward, ro.value, bootstrap=ro.bootstrap, **fl,
                              gamma=p["gamma"], lam=p["lam"])
        return {"advantages": adv, "returns": ret}
    if est == "vtrace":
        vs, pg = oracle.vtrace(ro.reward, ro.value, ro.log_rho, bootstrap=ro.bootstrap, **fl,
                               gamma=p["gamma"], lam=p["lam"], rho_bar=p["rho_bar"],
                               c_bar=p["c_bar"], pg_rho_bar=p["pg_rho_bar"])
        return {"vs": vs, "pg_advantages": pg}
    q = oracle.retrace(ro.reward, ro.q_taken, ro.expected_q, ro.rho, bootstrap_ev=ro.bootstrap,
                       **fl, gamma=p["gamma"], lam=p["lam"])
    return {"q_ret": q}


class Placed:
    """A [N, T] tensor inside a sentinel-filled buffer, with row stride ld and an element
    offset from a 256-byte aligned start (offset % 4 != 0 defeats 128-bit access)."""

    def __init__(self, a: np.ndarray | None, N, T, ld, offset, dtype, fill, device):
        n_el = GUARD + offset + max(N * ld, 1) + GUARD
        if device == "pinned":  # page-locked host memory, read and written in place
            self.buf = torch.full((n_el,), fill, dtype=dtype).pin_memory()
        else:
            self.buf = torch.full((n_el,), fill, dtype=dtype, device=device)
        self.lo = GUARD + offset
        self.view = self.buf[self.lo:self.lo + N * ld].view(N, ld)[:, :T]
        if a is not None:
            self.view.copy_(torch.from_numpy(np.ascontiguousarray(a)).to(dtype))
        self.N, self.T, self.ld = N, T, ld

    def untouched_outside(self, fill) -> bool:
        host = self.buf.cpu().numpy().copy()
        inner = host[self.lo:self.lo + self.N * self.ld].reshape(self.N, self.ld)
        inner[:, :self.T] = fill
        return bool(np.all(host == np.asarray(fill, dtype=host.dtype)))


def run_gpu(est, ro, params, ld=None, offset=0, bool_flags=False, device="cuda:0",
            check_guards=True, drop_second_output=False, workspace=None,
            in_dtype=torch.float32, host=None, out_offset=None):
    """Run `est` on the CUDA path; returns {output name: float64 array}. `workspace`
    (a zeroed uint8 CUDA tensor) selects the look-back (_ex) entry point; in_dtype
    torch.bfloat16 places the data inputs as bf16 (the _bf16 entry points). `host`
    ("all", "inputs" or "outputs") places those buffers in pinned host memory, which
    the kernels then read or write in place. `out_offset` places the outputs at another
    element offset than the inputs."""
    N, T = ro.N, ro.T
    in_dev = "pinned" if host in ("all", "inputs") else device
    out_dev = "pinned" if host in ("all", "outputs") else device
    ws = dict(workspace=workspace)
    ld = T if ld is None else ld
    p = dict(DEFAULT_PARAMS[est], **params)

    def f32(a):
        return None if a is None else Placed(a, N, T, ld, offset, in_dtype, 0.0, in_dev)

    def flag(a):
        if a is None:
            return None
        dt = torch.bool if bool_flags else torch.uint8
        return Placed(a.astype(bool) if bool_flags else a, N, T, ld, offset, dt, 1, in_dev)

    boot = None
    if ro.bootstrap is not None:
        boot = torch.from_numpy(ro.bootstrap)
        boot = boot.pin_memory() if in_dev == "pinned" else boot.to(device)
    r, term, trunc = f32(ro.reward), flag(ro.terminated), flag(ro.truncated)
    tv = f32(ro.trunc_value) if ro.truncated is not None else None
    out_off = offset if out_offset is None else out_offset
    outs = {name: Placed(None, N, T, ld, out_off, torch.float32, SENTINEL, out_dev)
            for name in OUTPUTS[est]}
    if drop_second_output and len(outs) == 2:
        outs.pop(OUTPUTS[est][1])
    v = lambda x: None if x is None else x.view
    fl = dict(terminated=term.view, truncated=v(trunc), trunc_value=v(tv))
    o = lambda name: v(outs.get(name))
    if est == "return":
        rlca.rlca_discounted_return(r.view, **fl, bootstrap=boot, gamma=p["gamma"],
                                    returns=o("returns"), **ws)
    elif est == "td_lambda":
        rlca.rlca_td_lambda(r.view, f32(ro.value).view, **fl, bootstrap=boot,
                            gamma=p["gamma"], lam=p["lam"], targets=o("targets"), **ws)
    elif est == "gae":
        rlca.rlca_gae(r.view, f32(ro.value).view, **fl, bootstrap=boot, gamma=p["gamma"],
                      lam=p["lam"], advantages=o("advantages"), returns=o("returns"),
                      want_returns=False, **ws)
    elif est == "vtrace":
        rlca.rlca_vtrace(r.view, f32(ro.value).view, f32(ro.log_rho).view, **fl,
                         bootstrap=boot, gamma=p["gamma"], lam=p["lam"], rho_bar=p["rho_bar"],
                         c_bar=p["c_bar"], pg_rho_bar=p["pg_rho_bar"], vs=o("vs"),
                         pg_advantages=o("pg_advantages"), want_pg=False, **ws)
    else:
        rlca.rlca_retrace(r.view, f32(ro.q_taken).view, f32(ro.expected_q).view,
                          f32(ro.rho).view, **fl, bootstrap_ev=boot, gamma=p["gamma"],
                          lam=p["lam"], q_ret=o("q_ret"), **ws)
    torch.cuda.synchronize()
    if check_guards:
        for name, pl in outs.items():
            assert pl.untouched_outside(SENTINEL), f"{est}: write outside {name}"
    return {name: pl.view.cpu().numpy().astype(np.float64) for name, pl in outs.items()}


def assert_parity(gpu: dict, ref: dict, what: str, tol=TOL):
    for name, g in gpu.items():
        r = ref[name]
        assert g.shape == r.shape, (what, name)
        nan_g, nan_r = np.isnan(g), np.isnan(r)
        assert np.array_equal(nan_g, nan_r), f"{what}/{name}: NaN pattern differs"
        fin = ~nan_r
        if not fin.any():
            continue
        assert np.array_equal(np.isinf(g[fin]), np.isinf(r[fin])), f"{what}/{name}: Inf"
        ok = np.isfinite(r)
        if not ok.any():
            continue
        err = np.max(np.abs(g[ok] - r[ok]))
        bound = tol * (1.0 + np.max(np.abs(r[ok])))
        assert err <= bound, f"{what}/{name}: max|err| {err:.3e} > {bound:.3e}"


def bf16_rounded(ro):
    """The rollout with every per-step data input rounded to bf16 (kept as fp32 arrays,
    so the oracle sees exactly the values the bf16 kernels widen)."""
    import copy
    out = copy.copy(ro)
    for k in ("reward", "value", "trunc_value", "log_rho", "q_taken", "expected_q", "rho"):
        a = getattr(ro, k)
        if a is not None:
            setattr(out, k, torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)
                    .to(torch.float32).numpy())
    return out


def fp16_rounded(ro):
    """The rollout with every per-step data input rounded to fp16 (round to nearest even,
    kept as fp32 arrays: fp16 values are exact in fp32)."""
    import copy
    out = copy.copy(ro)
    for k in ("reward", "value", "trunc_value", "log_rho", "q_taken", "expected_q", "rho"):
        a = getattr(ro, k)
        if a is not None:
            setattr(out, k, torch.from_numpy(np.ascontiguousarray(a)).to(torch.float16)
                    .to(torch.float32).numpy())
    return out
