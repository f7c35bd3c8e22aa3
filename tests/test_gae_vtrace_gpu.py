"""GPU parity of the fused GAE + V-trace call (one read of reward, value, log ratios and
flags; four outputs) against the fp64 oracle's separate GAE and V-trace loops, with the
same tolerance as the other parity tests. Covers whole-row tiles, one row per CTA, the
row loop, ragged tails, padded and offset layouts (with untouched guard zones), the
optional outputs, and buffers in pinned host memory."""
import numpy as np
import pytest
import torch

import oracle
import segmented_associative_scan_gb300 as rlca
import synthetic_rollouts as sr
from parity_helpers import SENTINEL, Placed, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    rlca.build()
    rlca.lib()


def run_pair(ro, p, ld=None, offset=0, device="cuda:0", drop=False):
    N, T = ro.N, ro.T
    ld = T if ld is None else ld
    f = lambda a: None if a is None else Placed(a, N, T, ld, offset, torch.float32, 0.0, device)
    fl = lambda a: None if a is None else Placed(a, N, T, ld, offset, torch.uint8, 1, device)
    out = lambda: Placed(None, N, T, ld, offset, torch.float32, SENTINEL, device)
    r, v, lr = f(ro.reward), f(ro.value), f(ro.log_rho)
    d, tr = fl(ro.terminated), fl(ro.truncated)
    tv = f(ro.trunc_value) if ro.truncated is not None else None
    boot = torch.from_numpy(ro.bootstrap)
    boot = boot.pin_memory() if device == "pinned" else boot.to(device)
    outs = {"adv": out(), "vs": out()}
    if not drop:
        outs["ret"], outs["pg"] = out(), out()
    view = lambda x: None if x is None else x.view
    rlca.rlca_gae_vtrace(r.view, v.view, lr.view, d.view, view(tr), view(tv), boot,
                         gamma=p["gamma"], lam=p["lam"], lam_vtrace=p["lam_v"],
                         rho_bar=p["rho_bar"], c_bar=p["c_bar"], pg_rho_bar=p["pg_rho_bar"],
                         advantages=outs["adv"].view, returns=view(outs.get("ret")),
                         vs=outs["vs"].view, pg_advantages=view(outs.get("pg")),
                         want_returns=not drop, want_pg=not drop)
    torch.cuda.synchronize()
    for name, pl in outs.items():
        assert pl.untouched_outside(SENTINEL), f"write outside {name}"
    return {k: pl.view.cpu().numpy().astype(np.float64) for k, pl in outs.items()}


def oracle_pair(ro, p):
    fl = dict(terminated=ro.terminated, truncated=ro.truncated, trunc_value=ro.trunc_value,
              bootstrap=ro.bootstrap)
    adv, ret = oracle.gae(ro.reward, ro.value, **fl, gamma=p["gamma"], lam=p["lam"])
    vs, pg = oracle.vtrace(ro.reward, ro.value, ro.log_rho, **fl, gamma=p["gamma"],
                           lam=p["lam_v"], rho_bar=p["rho_bar"], c_bar=p["c_bar"],
                           pg_rho_bar=p["pg_rho_bar"])
    return {"adv": adv, "ret": ret, "vs": vs, "pg": pg}


P = dict(gamma=0.99, lam=0.95, lam_v=1.0, rho_bar=1.0, c_bar=1.0, pg_rho_bar=1.0)


@pytest.mark.parametrize("N", [1, 5, 33])
@pytest.mark.parametrize("T", [1, 7, 128, 256, 300, 512, 1000, 1024, 1025, 3000])
def test_shape_grid(N, T):
    ro = sr.generic(N, T, seed=N * 31 + T, p_term=0.02, p_trunc=0.01)
    assert_parity(run_pair(ro, P), oracle_pair(ro, P), f"gae+vtrace N={N} T={T}")


@pytest.mark.parametrize("params", [dict(lam_v=0.9, c_bar=0.9, pg_rho_bar=1.3),
                                    dict(lam=0.0, rho_bar=0.8, c_bar=1.2),
                                    dict(lam=1.0, gamma=1.0)])
def test_parameters(params):
    ro = sr.generic(7, 1024, seed=11)
    p = dict(P, **params)
    assert_parity(run_pair(ro, p), oracle_pair(ro, p), f"gae+vtrace {params}")


@pytest.mark.parametrize("ld_extra,offset", [(0, 0), (8, 0), (4, 0), (0, 2), (3, 1)])
@pytest.mark.parametrize("T", [300, 1024, 2000])
def test_layouts(ld_extra, offset, T):
    ro = sr.generic(6, T, seed=T + ld_extra + offset)
    assert_parity(run_pair(ro, P, ld=T + ld_extra, offset=offset), oracle_pair(ro, P),
                  f"gae+vtrace T={T} ld+{ld_extra} off={offset}")


def test_optional_outputs_and_no_truncation():
    ro = sr.generic(9, 1024, seed=12, p_trunc=0.0)
    ro.truncated = None
    got = run_pair(ro, P, drop=True)
    assert set(got) == {"adv", "vs"}
    assert_parity(got, oracle_pair(ro, P), "gae+vtrace advantages and vs only")


def test_vtrace_workload_with_gae():
    ro = sr.vtrace()
    p = dict(P, gamma=0.99)
    assert_parity(run_pair(ro, p), oracle_pair(ro, p), "gae+vtrace 8192x256")


def test_pinned_host_buffers():
    ro = sr.generic(16, 1024, seed=13)
    assert_parity(run_pair(ro, P, device="pinned"), oracle_pair(ro, P), "gae+vtrace host")


@pytest.mark.parametrize("T", [13, 250, 1001, 3001])
def test_wide_access_with_ragged_tails(T):
    """Rows padded to a multiple of 8 floats (256-bit access) with a ragged last thread."""
    ro = sr.generic(11, T, seed=T + 29, p_term=0.02, p_trunc=0.01)
    assert_parity(run_pair(ro, P, ld=(T + 7) // 8 * 8), oracle_pair(ro, P),
                  f"gae+vtrace T={T}")
