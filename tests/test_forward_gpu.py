"""GPU parity of the forward scans (eligibility traces, episodic prefix sums) against
the fp64 oracle: shape grid with ragged tails and several rows per warp, flag patterns,
strided and unaligned layouts with guard zones, and exact NaN isolation."""
import numpy as np
import pytest
import torch

import oracle
import segmented_associative_scan_gb300 as rlca
import synthetic_rollouts as sr
from parity_helpers import SENTINEL, TOL, Placed, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    rlca.build()
    rlca.lib()


def run_both(ro, kind, decay=0.95, ld=None, offset=0, with_trunc=True, with_init=True):
    N, T = ro.N, ro.T
    ld = T if ld is None else ld
    dev = "cuda:0"
    x = Placed(ro.value, N, T, ld, offset, torch.float32, 0.0, dev)
    d = Placed(ro.terminated, N, T, ld, offset, torch.uint8, 1, dev)
    tr = Placed(ro.truncated, N, T, ld, offset, torch.uint8, 1, dev) if with_trunc else None
    init = torch.from_numpy(ro.bootstrap).to(dev) if with_init else None
    out = Placed(None, N, T, ld, offset, torch.float32, SENTINEL, dev)
    trn = tr.view if tr is not None else None
    if kind == "trace":
        rlca.rlca_eligibility_trace(x.view, d.view, trn, init, decay=decay, traces=out.view)
        ref = oracle.eligibility_trace(ro.value, ro.terminated,
                                       ro.truncated if with_trunc else None,
                                       ro.bootstrap if with_init else None, decay=decay)
    else:
        rlca.rlca_episodic_prefix_sum(x.view, d.view, trn, init, sums=out.view)
        ref = oracle.episodic_prefix_sum(ro.value, ro.terminated,
                                         ro.truncated if with_trunc else None,
                                         ro.bootstrap if with_init else None)
    torch.cuda.synchronize()
    assert out.untouched_outside(SENTINEL), "write outside the output block"
    return out.view.cpu().numpy().astype(np.float64), ref


T_GRID = [1, 2, 3, 7, 8, 9, 16, 31, 32, 33, 100, 255, 256, 257, 511, 512, 1000, 1024,
          1025, 4096, 5000]


@pytest.mark.parametrize("N", [1, 5, 70])
@pytest.mark.parametrize("T", T_GRID)
def test_forward_shape_grid(N, T):
    ro = sr.generic(N, T, seed=N * 7 + T, p_term=0.03, p_trunc=0.02)
    for kind in ("trace", "sum"):
        g, r = run_both(ro, kind)
        assert_parity({"o": g}, {"o": r}, f"{kind} N={N} T={T}")


@pytest.mark.parametrize("decay", [0.0, 0.5, 0.99, 1.0])
def test_forward_decays_and_options(decay):
    ro = sr.generic(9, 1300, seed=3, p_term=0.01, p_trunc=0.01)
    for with_trunc in (True, False):
        for with_init in (True, False):
            g, r = run_both(ro, "trace", decay=decay, with_trunc=with_trunc,
                            with_init=with_init)
            assert_parity({"o": g}, {"o": r}, f"decay={decay} {with_trunc} {with_init}")


@pytest.mark.parametrize("pattern", ["all_done", "none", "done_at_0", "done_at_last",
                                     "every_other"])
def test_forward_flag_patterns(pattern):
    ro = sr.generic(6, 777, seed=4)
    term = np.zeros_like(ro.terminated)
    if pattern == "all_done":
        term[:] = 1
    elif pattern == "done_at_0":
        term[:, 0] = 1
    elif pattern == "done_at_last":
        term[:, -1] = 1
    elif pattern == "every_other":
        term[:, ::2] = 1
    ro.terminated = term
    ro.truncated = np.zeros_like(term)
    for kind in ("trace", "sum"):
        g, r = run_both(ro, kind)
        assert_parity({"o": g}, {"o": r}, f"{kind} {pattern}")


@pytest.mark.parametrize("ld_extra,offset", [(0, 0), (4, 0), (3, 0), (0, 1), (5, 3)])
@pytest.mark.parametrize("T", [12, 256, 1500])
def test_forward_layouts(ld_extra, offset, T):
    ro = sr.generic(3, T, seed=5 + T)
    for kind in ("trace", "sum"):
        g, r = run_both(ro, kind, ld=T + ld_extra, offset=offset)
        assert_parity({"o": g}, {"o": r}, f"{kind} ld=T+{ld_extra} off={offset}")


@pytest.mark.parametrize("T", [200, 3000])
def test_forward_nan_stays_in_its_episode(T):
    ro = sr.generic(3, T, seed=6, p_term=0.01, p_trunc=0.01)
    clean, _ = run_both(ro, "trace")
    n, k = 2, T // 2
    ro.value[n, k] = np.nan
    dirty, _ = run_both(ro, "trace")
    e = k
    while e + 1 < T and not (ro.terminated[n, e] or ro.truncated[n, e]):
        e += 1
    a, b = clean.copy(), dirty.copy()
    a[n, k:e + 1] = b[n, k:e + 1] = 0.0
    assert np.array_equal(a, b)
    assert np.isnan(dirty[n, k:e + 1]).all()


def test_forward_workload_sizes():
    """Full-size rollouts shaped like the bench workload and the long Retrace one."""
    for N, T in ((4096, 1024), (2048, 4096)):
        ro = sr.generic(N, T, seed=8, p_term=0.005, p_trunc=0.002)
        for kind in ("trace", "sum"):
            g, r = run_both(ro, kind)
            assert_parity({"o": g}, {"o": r}, f"{kind} {N}x{T}")


@pytest.mark.parametrize("kind", ["trace", "prefix_sum"])
@pytest.mark.parametrize("T", [13, 250, 1001, 3001])
def test_wide_access_with_ragged_tails(kind, T):
    """Rows padded to a multiple of 8 floats (256-bit access) with a ragged last thread."""
    ro = sr.generic(11, T, seed=T + 17, p_term=0.02, p_trunc=0.01)
    got, ref = run_both(ro, kind, ld=(T + 7) // 8 * 8)
    assert_parity({"o": got}, {"o": ref}, f"{kind} T={T}")


@pytest.mark.parametrize("N", [1, 6, 37])
@pytest.mark.parametrize("T", [260, 264, 500, 512, 520, 768, 1000, 1016, 1024])
def test_forward_pipelined_rows(N, T):
    """Rows of 257-1024 steps in 16-byte aligned rows: a warp per row walks its chunks of
    256 steps from the first with the next chunks' loads in flight; a ragged last chunk is
    loaded plainly at the end. Episode ends planted on the last step of a chunk (the next
    chunk starts afresh) and on the first step of one. (fp32 rows that one wave of warps
    holds keep three chunks in flight; more rows keep two: see the next test.)"""
    ro = sr.generic(N, T, seed=300 + 7 * N + T, p_term=0.01, p_trunc=0.01)
    for t in (255, 256, 511, 767):
        if t < T:
            ro.terminated[0, t] = 1
            ro.truncated[N - 1, t] = 1 - ro.terminated[N - 1, t]
    for kind in ("trace", "sum"):
        g, r = run_both(ro, kind)
        assert_parity({"o": g}, {"o": r}, f"{kind} N={N} T={T}")
        g, r = run_both(ro, kind, with_trunc=False, with_init=False)
        assert_parity({"o": g}, {"o": r}, f"{kind} N={N} T={T} no trunc, no init")


@pytest.mark.parametrize("ld_extra,offset", [(4, 0), (8, 0), (0, 4), (12, 8)])
@pytest.mark.parametrize("T", [264, 1000, 1024])
def test_forward_pipelined_layouts(T, ld_extra, offset):
    ro = sr.generic(9, T, seed=400 + T + ld_extra + offset, p_term=0.01, p_trunc=0.01)
    for kind in ("trace", "sum"):
        g, r = run_both(ro, kind, ld=T + ld_extra, offset=offset)
        assert_parity({"o": g}, {"o": r}, f"{kind} T={T} ld+{ld_extra} off={offset}")


@pytest.mark.parametrize("N,T", [(2600, 1024), (3000, 1024), (4096, 600), (4256, 777),
                                 (4400, 1024), (6000, 520)])
def test_forward_pipelined_rows_by_grid_size(N, T):
    """fp32 rows whose grid fills most of one wave of warps under the 7-CTA cap take three
    chunks in flight ([3000, 1024], [4096, 600], [4256, 777]); fewer rows ([2600, 1024])
    and more than one wave ([4400, 1024], [6000, 520]) two chunks and no cap."""
    ro = sr.generic(N, T, seed=500 + N + T, p_term=0.01, p_trunc=0.01)
    for kind in ("trace", "sum"):
        g, r = run_both(ro, kind)
        assert_parity({"o": g}, {"o": r}, f"{kind} N={N} T={T}")
