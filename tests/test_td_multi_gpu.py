"""GPU parity of the fused multi-lambda TD(lambda): every output equals the oracle's
TD(lambda) for its lambda (lambda = 1 is the discounted return), on the [4096,128]
workload's lambdas and on a shape grid that covers whole-row tiles and the row loop."""
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


def run(ro, lams, gamma=0.99, ld=None, offset=0):
    N, T = ro.N, ro.T
    ld = T if ld is None else ld
    dev = "cuda:0"
    f = lambda a: Placed(a, N, T, ld, offset, torch.float32, 0.0, dev)
    fl = lambda a: None if a is None else Placed(a, N, T, ld, offset, torch.uint8, 1, dev)
    tr = fl(ro.truncated)
    tv = f(ro.trunc_value) if ro.truncated is not None else None
    outs = [Placed(None, N, T, ld, offset, torch.float32, SENTINEL, dev) for _ in lams]
    boot = torch.from_numpy(ro.bootstrap).to(dev) if ro.bootstrap is not None else None
    rlca.rlca_td_lambda_multi(f(ro.reward).view, f(ro.value).view, fl(ro.terminated).view,
                              tr.view if tr else None, tv.view if tv else None, boot,
                              gamma=gamma, lams=lams, targets=[o.view for o in outs])
    torch.cuda.synchronize()
    got = []
    for o in outs:
        assert o.untouched_outside(SENTINEL)
        got.append(o.view.cpu().numpy().astype(np.float64))
    return got


def test_workload_return_td_4096x128():
    ro = sr.return_td()
    lams = ro.params["lams"]
    got = run(ro, lams, gamma=ro.params["gamma"])
    for g, lam in zip(got, lams):
        ref = oracle.td_lambda(ro.reward, ro.value, ro.terminated, bootstrap=ro.bootstrap,
                               gamma=ro.params["gamma"], lam=lam)
        assert_parity({"t": g}, {"t": ref}, f"lambda={lam}")
    ref_ret = oracle.discounted_return(ro.reward, ro.terminated, bootstrap=ro.bootstrap,
                                       gamma=ro.params["gamma"])
    assert_parity({"t": got[2]}, {"t": ref_ret}, "lambda=1 is the discounted return")


@pytest.mark.parametrize("T", [1, 5, 128, 257, 1000, 1024, 1025, 3000])
@pytest.mark.parametrize("k", [1, 2, 4])
def test_shapes_and_counts(T, k):
    ro = sr.generic(6, T, seed=T + k, p_term=0.02, p_trunc=0.02)
    lams = [0.0, 0.95, 0.5, 1.0][:k]
    got = run(ro, lams)
    for g, lam in zip(got, lams):
        ref = oracle.td_lambda(ro.reward, ro.value, ro.terminated, ro.truncated,
                               ro.trunc_value, ro.bootstrap, gamma=0.99, lam=lam)
        assert_parity({"t": g}, {"t": ref}, f"T={T} lambda={lam}")


@pytest.mark.parametrize("ld_extra,offset", [(3, 0), (0, 1), (4, 0)])
def test_layouts(ld_extra, offset):
    ro = sr.generic(5, 700, seed=9)
    lams = [0.3, 0.9, 1.0]
    got = run(ro, lams, ld=700 + ld_extra, offset=offset)
    for g, lam in zip(got, lams):
        ref = oracle.td_lambda(ro.reward, ro.value, ro.terminated, ro.truncated,
                               ro.trunc_value, ro.bootstrap, gamma=0.99, lam=lam)
        assert_parity({"t": g}, {"t": ref}, f"lambda={lam}")


def test_full_size_4096x1024():
    ro = sr.generic(4096, 1024, seed=10, p_term=0.02, p_trunc=0.0)
    ro.truncated = None
    lams = [0.0, 0.9, 1.0]
    got = run(ro, lams)
    for g, lam in zip(got, lams):
        ref = oracle.td_lambda(ro.reward, ro.value, ro.terminated, bootstrap=ro.bootstrap,
                               gamma=0.99, lam=lam)
        assert_parity({"t": g}, {"t": ref}, f"lambda={lam}")


@pytest.mark.parametrize("T", [13, 250, 1001, 3001])
def test_wide_access_with_ragged_tails(T):
    """Rows padded to a multiple of 8 floats (256-bit access) with a ragged last thread."""
    ro = sr.generic(11, T, seed=T + 23, p_term=0.02, p_trunc=0.01)
    lams = [0.0, 0.9, 1.0]
    got = run(ro, lams, ld=(T + 7) // 8 * 8)
    for g, lam in zip(got, lams):
        ref = oracle.td_lambda(ro.reward, ro.value, ro.terminated, ro.truncated,
                               ro.trunc_value, ro.bootstrap, gamma=0.99, lam=lam)
        assert_parity({"t": g}, {"t": ref}, f"td multi lambda={lam} T={T}")


@pytest.mark.parametrize("trunc", [True, False])
@pytest.mark.parametrize("T", [513, 520, 777, 1000, 1016, 1023, 1024])
def test_pipelined_rows(T, trunc):
    """Rows of 513-1024 steps take the pipelined warp rows (a warp per row with the next
    chunk's loads in flight): 3-4 chunks per row, ragged first chunks, with and without
    truncation, one to four lambdas."""
    ro = sr.generic(37, T, seed=6000 + T, p_term=0.01, p_trunc=0.01 if trunc else 0.0)
    if not trunc:
        ro.truncated = None
    for lams in ([0.9], [0.0, 0.9, 1.0], [0.0, 0.5, 0.95, 1.0]):
        got = run(ro, lams)
        for g, lam in zip(got, lams):
            ref = oracle.td_lambda(ro.reward, ro.value, ro.terminated, ro.truncated,
                                   ro.trunc_value, ro.bootstrap, gamma=0.99, lam=lam)
            assert_parity({"t": g}, {"t": ref}, f"T={T} lambdas={lams} lambda={lam}")


@pytest.mark.parametrize("ld_extra,offset", [(4, 0), (0, 4), (8, 0), (3, 0)])
def test_pipelined_rows_layouts(ld_extra, offset):
    """128-bit rows (ld % 8 == 4, a 16-byte offset), 32-byte rows, and an odd ld, which
    leaves the pipeline for the scalar CTA tiles."""
    ro = sr.generic(9, 1000, seed=6100 + ld_extra + offset, p_term=0.01, p_trunc=0.01)
    lams = [0.0, 0.9, 1.0]
    got = run(ro, lams, ld=1000 + ld_extra, offset=offset)
    for g, lam in zip(got, lams):
        ref = oracle.td_lambda(ro.reward, ro.value, ro.terminated, ro.truncated,
                               ro.trunc_value, ro.bootstrap, gamma=0.99, lam=lam)
        assert_parity({"t": g}, {"t": ref}, f"ld+{ld_extra} off={offset} lambda={lam}")
